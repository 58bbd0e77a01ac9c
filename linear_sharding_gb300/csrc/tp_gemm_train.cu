// tp_gemm_train.cu - launches of the tensor-core GEMM (tp_gemm_impl.cuh) for
// the training epilogues (the column-parallel GEMM that also keeps its
// pre-activations for the backward pass; the backward GEMM dH = dZ W2^T with
// the activation's derivative fused into its epilogue) and for the
// transformer block (the head-major QKV projection, and the row-parallel
// projections with their residual adds fused); plus the bf16 transpose
// that gives the weight-gradient and attention GEMMs K-major operands.
#include "tp_gemm_impl.cuh"

namespace tp {

using namespace gemm_impl;

cudaError_t launch_gemm_train(GemmCfg cfg, Epi epi, const CUtensorMap &mapA, const CUtensorMap &mapB,
                              const GemmArgs &args, int num_sms, cudaStream_t stream) {
  switch (cfg) {
    case CFG_PAIR_N256:
      switch (epi) {
        case EPI_GELU_SAVE_BF16: return launch_pair<EPI_GELU_SAVE_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_SWIGLU_SAVE_BF16:
          return launch_pair<EPI_SWIGLU_SAVE_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_DGELU_BF16: return launch_pair<EPI_DGELU_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_DSWIGLU_BF16: return launch_pair<EPI_DSWIGLU_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_QKV_HEADS_BF16: return launch_pair<EPI_QKV_HEADS_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_F32_RESID: return launch_pair<EPI_F32_RESID>(mapA, mapB, args, num_sms, stream);
        case EPI_F32_MN: return launch_pair<EPI_F32_MN>(mapA, mapB, args, num_sms, stream);
        default: break;
      }
      break;
    case CFG_N256:
      switch (epi) {
        case EPI_GELU_SAVE_BF16: return launch_impl<256, EPI_GELU_SAVE_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_SWIGLU_SAVE_BF16:
          return launch_impl<256, EPI_SWIGLU_SAVE_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_DGELU_BF16: return launch_impl<256, EPI_DGELU_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_DSWIGLU_BF16: return launch_impl<256, EPI_DSWIGLU_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_QKV_HEADS_BF16:
          return launch_impl<256, EPI_QKV_HEADS_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_F32_RESID: return launch_impl<256, EPI_F32_RESID>(mapA, mapB, args, num_sms, stream);
        case EPI_F32_MN: return launch_impl<256, EPI_F32_MN>(mapA, mapB, args, num_sms, stream);
        default: break;
      }
      break;
    case CFG_N128:
      switch (epi) {
        case EPI_GELU_SAVE_BF16: return launch_impl<128, EPI_GELU_SAVE_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_DGELU_BF16: return launch_impl<128, EPI_DGELU_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_DSWIGLU_BF16: return launch_impl<128, EPI_DSWIGLU_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_QKV_HEADS_BF16:
          return launch_impl<128, EPI_QKV_HEADS_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_F32_RESID: return launch_impl<128, EPI_F32_RESID>(mapA, mapB, args, num_sms, stream);
        case EPI_F32_MN: return launch_impl<128, EPI_F32_MN>(mapA, mapB, args, num_sms, stream);
        default: break;
      }
      break;
    default:
      break;
  }
  return cudaErrorInvalidValue;
}

namespace {

// 64 x 64 tiles.  Thread t of 256 reads 8 elements (16 bytes) of source rows 2i and
// 2i + 1, i = t / 8, columns 8 (t % 8) ..; pairs them by column (__byte_perm) into
// 32-bit words w = (src[2i][c], src[2i + 1][c]), stored at T[c][i] (pitch 33 words:
// at most two-way bank conflicts); destination row c then reads its words T[c][8q ..]
// (conflict-free) and writes 16 elements (two 16-byte stores).  Every warp reads and
// writes whole 128-byte lines.  Source rows past `rows` read as zero (the padding);
// unaligned or partial groups take element-wise loads and stores.
__global__ void __launch_bounds__(256) transpose_pad_kernel(const uint16_t *src, long long rows, long long cols,
                                                            long long src_ld, long long src_batch, uint16_t *dst,
                                                            long long dst_ld, long long dst_batch, int vec_ok) {
  __shared__ uint32_t T[64][33];
  const int b = blockIdx.z;
  const long long r0 = static_cast<long long>(blockIdx.x) * 64;  // source rows = destination columns
  const long long c0 = static_cast<long long>(blockIdx.y) * 64;  // source columns = destination rows
  const uint16_t *s = src + b * src_batch;
  uint16_t *d = dst + b * dst_batch;
  {
    const int i = threadIdx.x >> 3, g = threadIdx.x & 7;
    const long long c = c0 + 8 * g;
    uint32_t w0[4] = {0u, 0u, 0u, 0u}, w1[4] = {0u, 0u, 0u, 0u};  // rows 2i and 2i + 1, 8 elements each
    for (int h = 0; h < 2; ++h) {
      const long long r = r0 + 2 * i + h;
      uint32_t *w = h ? w1 : w0;
      if (r >= rows) continue;
      const uint16_t *p = s + r * src_ld + c;
      if (vec_ok && c + 8 <= cols) {
        const uint4 v = *reinterpret_cast<const uint4 *>(p);
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        w[3] = v.w;
      } else {
        for (int e = 0; e < 8; ++e)
          if (c + e < cols) w[e >> 1] |= static_cast<uint32_t>(p[e]) << (16 * (e & 1));
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // columns 8g + 2k (low halves) and 8g + 2k + 1 (high halves), rows 2i / 2i + 1
      T[8 * g + 2 * k][i] = __byte_perm(w0[k], w1[k], 0x5410);
      T[8 * g + 2 * k + 1][i] = __byte_perm(w0[k], w1[k], 0x7632);
    }
  }
  __syncthreads();
  {
    const int cr = threadIdx.x >> 2, q = threadIdx.x & 3;
    const long long c = c0 + cr;                // destination row
    const long long r = r0 + 16 * q;            // first destination column
    if (c >= cols || r >= dst_ld) return;
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = T[cr][8 * q + k];
    uint16_t *p = d + c * dst_ld + r;
    if (vec_ok && r + 16 <= dst_ld) {
      reinterpret_cast<uint4 *>(p)[0] = make_uint4(w[0], w[1], w[2], w[3]);
      reinterpret_cast<uint4 *>(p)[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
      for (int e = 0; e < 16 && r + e < dst_ld; ++e) p[e] = static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1)));
    }
  }
}

}  // namespace

cudaError_t launch_transpose_pad(const void *src, long long rows, long long cols, long long src_ld,
                                 long long src_batch, void *dst, long long dst_ld, long long dst_batch,
                                 int batch, cudaStream_t stream) {
  if (rows < 0 || cols < 0 || dst_ld < rows || batch < 1 || batch > 65535) return cudaErrorInvalidValue;
  if (cols == 0 || dst_ld == 0) return cudaSuccess;
  const long long gx = (dst_ld + 63) / 64, gy = (cols + 63) / 64;
  if (gy > 65535 || gx > 2147483647LL) return cudaErrorInvalidValue;
  // 16-byte accesses when every row (and batch) of both sides starts 16-byte aligned
  const bool vec_ok = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && (reinterpret_cast<uintptr_t>(dst) % 16 == 0) &&
                      src_ld % 8 == 0 && dst_ld % 8 == 0 && src_batch % 8 == 0 && dst_batch % 8 == 0;
  transpose_pad_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), batch), 256, 0, stream>>>(
      static_cast<const uint16_t *>(src), rows, cols, src_ld, src_batch, static_cast<uint16_t *>(dst), dst_ld,
      dst_batch, vec_ok ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace tp
