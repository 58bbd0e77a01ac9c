// tp_gemm_train.cu - launches of the tensor-core GEMM (tp_gemm_impl.cuh) for
// the training epilogues (the column-parallel GEMM that also keeps its
// pre-activations for the backward pass; the backward GEMM dH = dZ W2^T with
// the activation's derivative fused into its epilogue) and for the
// transformer block's head-major QKV projection; plus the bf16 transpose
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
        default: break;
      }
      break;
    default:
      break;
  }
  return cudaErrorInvalidValue;
}

namespace {

// 32 x 32 tiles through shared memory: reads run along the source rows'
// columns, writes along the destination rows; padding columns are zeroed.
__global__ void transpose_pad_kernel(const uint16_t *src, long long rows, long long cols, long long src_ld,
                                     long long src_batch, uint16_t *dst, long long dst_ld,
                                     long long dst_batch) {
  __shared__ uint16_t tile[32][33];
  const int b = blockIdx.z;
  const long long c0 = static_cast<long long>(blockIdx.y) * 32;  // source column = dst row
  const long long r0 = static_cast<long long>(blockIdx.x) * 32;  // source row = dst column
  const uint16_t *s = src + b * src_batch;
  uint16_t *d = dst + b * dst_batch;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const long long r = r0 + i, c = c0 + threadIdx.x;
    tile[i][threadIdx.x] = (r < rows && c < cols) ? s[r * src_ld + c] : static_cast<uint16_t>(0);
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const long long c = c0 + i, r = r0 + threadIdx.x;
    if (c < cols && r < dst_ld) d[c * dst_ld + r] = tile[threadIdx.x][i];
  }
}

}  // namespace

cudaError_t launch_transpose_pad(const void *src, long long rows, long long cols, long long src_ld,
                                 long long src_batch, void *dst, long long dst_ld, long long dst_batch,
                                 int batch, cudaStream_t stream) {
  if (rows < 0 || cols < 0 || dst_ld < rows || batch < 1 || batch > 65535) return cudaErrorInvalidValue;
  if (cols == 0 || dst_ld == 0) return cudaSuccess;
  const long long gx = (dst_ld + 31) / 32, gy = (cols + 31) / 32;
  if (gy > 65535 || gx > 2147483647LL) return cudaErrorInvalidValue;
  transpose_pad_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), batch), dim3(32, 8), 0,
                         stream>>>(static_cast<const uint16_t *>(src), rows, cols, src_ld, src_batch,
                                   static_cast<uint16_t *>(dst), dst_ld, dst_batch);
  return cudaGetLastError();
}

}  // namespace tp
