// tp_kernels.cu - the non-tensor-core kernels of the tensor-parallel MLP:
//   - the shard-sum, i.e. the all-reduce-sum Z = sum_i Z_i done as
//     arithmetic in device memory ("Slice the matrix itself", section
//     "Mathematical formulation - row-parallel matrix multiplication
//     summation"): float32, shards in ascending order, streaming 16-byte
//     loads and stores, grid sized to the SM count;
//   - the weight packing into per-shard K-major buffers (the column blocks
//     of W1 and row blocks of W2 of "Tensor Parallelism in Action", section
//     1; bfloat16 in k-tiles of 64) and its inverse for layout checks;
//   - the float32 CUDA-core GEMM used for float32 inputs;
//   - the decode activation, which finishes split-K first-layer partials.
#include <cuda_bf16.h>

#include <utility>

#include "tp_device.cuh"
#include "tp_internal.h"

namespace tp {
namespace {

__device__ __forceinline__ float gelu_erf(float x) {
  return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + __expf(-g)); }

// ---- shard-sum ----------------------------------------------------------

constexpr int kMaxParts = 64;

struct PartList {
  const float *p[kMaxParts];
};

__device__ __forceinline__ void add4(float4 &s, const float4 &v) {
  s.x += v.x;
  s.y += v.y;
  s.z += v.z;
  s.w += v.w;
}

// T known at compile time: all T 16-byte loads of an element group are in
// flight before the first add.
template <int T>
__global__ void __launch_bounds__(256) shard_sum_fixed(const PartList L, long long n4, float *Z) {
  pdl_trigger();
  pdl_wait();  // the partials come from the kernel before
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += stride) {
    float4 v[T];
#pragma unroll
    for (int t = 0; t < T; ++t) v[t] = __ldcs(reinterpret_cast<const float4 *>(L.p[t]) + i);
    float4 s = v[0];
#pragma unroll
    for (int t = 1; t < T; ++t) add4(s, v[t]);
    __stcs(reinterpret_cast<float4 *>(Z) + i, s);
  }
}

// Any T: groups of 8 loads in flight, added in ascending order.
__global__ void __launch_bounds__(256) shard_sum_any(const PartList L, int T, long long n4, float *Z) {
  pdl_trigger();
  pdl_wait();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += stride) {
    float4 s = __ldcs(reinterpret_cast<const float4 *>(L.p[0]) + i);
    for (int t0 = 1; t0 < T; t0 += 8) {
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (t0 + j < T) v[j] = __ldcs(reinterpret_cast<const float4 *>(L.p[t0 + j]) + i);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (t0 + j < T) add4(s, v[j]);
    }
    __stcs(reinterpret_cast<float4 *>(Z) + i, s);
  }
}

// Scalar path for elements [first, n) (the tail after the vector part, or
// everything when a pointer is not 16-byte aligned).
__global__ void shard_sum_scalar(const PartList L, int T, long long first, long long n, float *Z) {
  pdl_trigger();
  pdl_wait();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = first + static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    float s = L.p[0][i];
    for (int t = 1; t < T; ++t) s += L.p[t][i];
    Z[i] = s;
  }
}

// ---- reduce-scatter, all-gather, bf16 all-reduce ----------------------------

struct OutList {
  float *p[kMaxParts];
};

// out[i][k] = sum over t ascending of P_t[i nb + k], 16-byte groups
// (nb4 = nb / 4 groups per block).
__global__ void __launch_bounds__(256) reduce_scatter_vec(const PartList L, int T, const OutList O,
                                                          long long nb4, long long n4) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += stride) {
    float4 s = __ldcs(reinterpret_cast<const float4 *>(L.p[0]) + i);
    for (int t0 = 1; t0 < T; t0 += 8) {
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (t0 + j < T) v[j] = __ldcs(reinterpret_cast<const float4 *>(L.p[t0 + j]) + i);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (t0 + j < T) add4(s, v[j]);
    }
    const long long blk = i / nb4;
    __stcs(reinterpret_cast<float4 *>(O.p[blk]) + (i - blk * nb4), s);
  }
}

__global__ void reduce_scatter_scalar(const PartList L, int T, const OutList O, long long nb,
                                      long long n) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    float s = L.p[0][i];
    for (int t = 1; t < T; ++t) s += L.p[t][i];
    const long long blk = i / nb;
    O.p[blk][i - blk * nb] = s;
  }
}

struct ConstList {
  const uint8_t *p[kMaxParts];
};

// out[i nb_bytes + k] = parts[i][k]; 16-byte vectors when every block allows.
__global__ void all_gather_vec(const ConstList L, int T, long long nb16, uint4 *out) {
  const long long n16 = nb16 * T;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += stride) {
    const long long blk = i / nb16;
    const uint4 *src = reinterpret_cast<const uint4 *>(L.p[blk]);
    if (src == out + blk * nb16) continue;  // this block is already in place
    out[i] = __ldcs(src + (i - blk * nb16));
  }
}

__global__ void all_gather_bytes(const ConstList L, int T, long long nb_bytes, uint8_t *out) {
  const long long n = nb_bytes * T;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    const long long blk = i / nb_bytes;
    if (L.p[blk] == out + blk * nb_bytes) continue;
    out[i] = L.p[blk][i - blk * nb_bytes];
  }
}

// Z[k] = bf16(sum over t ascending of P_t[k]), 4 values per thread step.
__global__ void __launch_bounds__(256) shard_sum_bf16_vec(const PartList L, int T, long long n4,
                                                          __nv_bfloat16 *Z) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += stride) {
    float4 s = __ldcs(reinterpret_cast<const float4 *>(L.p[0]) + i);
    for (int t0 = 1; t0 < T; t0 += 8) {
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (t0 + j < T) v[j] = __ldcs(reinterpret_cast<const float4 *>(L.p[t0 + j]) + i);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (t0 + j < T) add4(s, v[j]);
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(s.x, s.y), hi = __floats2bfloat162_rn(s.z, s.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t *>(&lo);
    pk.y = *reinterpret_cast<uint32_t *>(&hi);
    reinterpret_cast<uint2 *>(Z)[i] = pk;
  }
}

__global__ void shard_sum_bf16_scalar(const PartList L, int T, long long first, long long n,
                                      __nv_bfloat16 *Z) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = first + static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    float s = L.p[0][i];
    for (int t = 1; t < T; ++t) s += L.p[t][i];
    Z[i] = __float2bfloat16_rn(s);
  }
}

// ---- residual stream ----------------------------------------------------------------

// h = x + z (x bf16, z float32) -> h float32 and its bf16 copy hb.
__global__ void residual_kernel(const __nv_bfloat16 *x, const float *z, float *h, __nv_bfloat16 *hb,
                                long long n) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float v = __bfloat162float(x[i]) + z[i];
    h[i] = v;
    hb[i] = __float2bfloat16_rn(v);
  }
}

__global__ void add_inplace_kernel(float *out, const float *h, long long n) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    out[i] += h[i];
}

// ---- packing ------------------------------------------------------------

template <typename E>
__device__ __forceinline__ void pack_src(int mode, int s, long long r, long long k, long long K,
                                         long long F, long long H, long long W, long long &srow,
                                         long long &scol) {
  switch (mode) {
    case PACK_W1:
      srow = k;
      scol = s * W + r;
      break;
    case PACK_W1_SWIGLU: {
      const long long blk = r / (2 * kSwigluGranule), off = r % (2 * kSwigluGranule);
      srow = k;
      scol = (off < kSwigluGranule ? 0 : F) + s * W + blk * kSwigluGranule + (off % kSwigluGranule);
      break;
    }
    case PACK_QKV:
      srow = k;
      scol = (r / W) * H + s * W + (r % W);
      break;
    default:  // PACK_ROWS
      srow = s * K + k;
      scol = r;
      break;
  }
}

// Offset of logical element [s][r][k] (S segments of R rows and K columns)
// in a packed buffer.  Row-major: (s R + r) K + k.  K-tile blocked: 64-wide
// k-tiles, each holding its 64 values of every row of the tensor map's view
// contiguously.  The first-layer modes view the buffer as S R rows of K
// (shards side by side along the rows), so tile kt is [S R][64] at
// kt S R 64; PACK_ROWS views it as R rows of K per shard (shards along K), so
// tile kt of shard s is [R][64] at (s K/64 + kt) R 64.
__device__ __forceinline__ long long packed_index(int mode, bool blocked, int s, int S, long long r,
                                                  long long R, long long k, long long K) {
  if (!blocked) return (static_cast<long long>(s) * R + r) * K + k;
  const long long kt = k >> 6, kk = k & 63;
  if (mode == PACK_ROWS) return ((static_cast<long long>(s) * (K >> 6) + kt) * R + r) * 64 + kk;
  return (kt * S * R + static_cast<long long>(s) * R + r) * 64 + kk;
}

// dst[s][r][k] = src[srow][scol] through a 32 x 32 shared-memory tile so that
// both the reads (along source columns) and the writes (along k) coalesce.
template <typename E>
__global__ void pack_kernel(int mode, bool blocked, const E *src, long long src_ld, E *dst, long long R,
                            long long K, long long F, long long H, long long W) {
  __shared__ E tile[32][33];
  const int s = blockIdx.z;
  const long long r0 = static_cast<long long>(blockIdx.y) * 32;
  const long long k0 = static_cast<long long>(blockIdx.x) * 32;
  for (int kk = threadIdx.y; kk < 32; kk += blockDim.y) {
    const long long k = k0 + kk, r = r0 + threadIdx.x;
    if (k < K && r < R) {
      long long srow, scol;
      pack_src<E>(mode, s, r, k, K, F, H, W, srow, scol);
      tile[kk][threadIdx.x] = src[srow * src_ld + scol];
    }
  }
  __syncthreads();
  for (int rr = threadIdx.y; rr < 32; rr += blockDim.y) {
    const long long r = r0 + rr, k = k0 + threadIdx.x;
    if (k < K && r < R) dst[packed_index(mode, blocked, s, gridDim.z, r, R, k, K)] = tile[threadIdx.x][rr];
  }
}

// Logical shard s from the packed buffer (layout checks only; one element
// per thread).  W1-like modes: out [K x Wl] with Wl = W (3W for QKV);
// PACK_ROWS: out [K x R].
template <typename E>
__global__ void unpack_kernel(int mode, bool blocked, const E *packed, E *out, int s, int S, int which,
                              long long R, long long K, long long W) {
  const long long cols = (mode == PACK_ROWS) ? R : (mode == PACK_QKV ? 3 * W : W);
  const long long total = K * cols;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long k = e / cols, c = e % cols;
    long long r;
    if (mode == PACK_W1_SWIGLU)
      r = (c / kSwigluGranule) * (2 * kSwigluGranule) + (which ? kSwigluGranule : 0) +
          c % kSwigluGranule;
    else
      r = c;
    out[e] = packed[packed_index(mode, blocked, s, S, r, R, k, K)];
  }
}

// ---- float32 CUDA-core GEMM ---------------------------------------------

constexpr int kSimtTile = 16;

// One thread per output (a gate/up pair for SwiGLU).  out column j maps to
// B row j (or gate row / up row of the packed SwiGLU layout).
__global__ void simt_gemm_kernel(const SimtArgs a) {
  __shared__ float As[kSimtTile][kSimtTile + 1];
  __shared__ float Bs[kSimtTile][kSimtTile + 1];
  __shared__ float Us[kSimtTile][kSimtTile + 1];
  const bool swiglu = a.epi == EPI_SWIGLU_BF16;
  const int n_out = swiglu ? a.N / 2 : a.N;
  const int m0 = blockIdx.y * kSimtTile, j0 = blockIdx.x * kSimtTile;
  const int slot = blockIdx.z;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int m = m0 + ty, j = j0 + tx;
  auto brow = [&](int jj) -> long long {
    if (!swiglu) return jj;
    return static_cast<long long>(jj / kSwigluGranule) * (2 * kSwigluGranule) + jj % kSwigluGranule;
  };
  float acc = 0.f, accu = 0.f;
  const int seg0 = slot * a.segs_per_slot;
  const int seg1 = min(a.nseg, seg0 + a.segs_per_slot);
  for (int seg = seg0; seg < seg1; ++seg) {
    for (int k0 = 0; k0 < a.k_seg; k0 += kSimtTile) {
      {  // A tile: rows m0.., cols k0..
        const int mm = m0 + ty, kk = k0 + tx;
        As[ty][tx] = (mm < a.M && kk < a.k_seg) ? a.A[mm * a.lda + seg * a.a_seg + kk] : 0.f;
        const int jj = j0 + ty;
        const bool ok = jj < n_out && kk < a.k_seg;
        Bs[ty][tx] = ok ? a.B[brow(jj) * a.ldb + seg * a.b_seg + kk] : 0.f;
        if (swiglu)
          Us[ty][tx] = ok ? a.B[(brow(jj) + kSwigluGranule) * a.ldb + seg * a.b_seg + kk] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < kSimtTile; ++kk) {
        acc = fmaf(As[ty][kk], Bs[tx][kk], acc);
        if (swiglu) accu = fmaf(As[ty][kk], Us[tx][kk], accu);
      }
      __syncthreads();
    }
  }
  if (m >= a.M || j >= n_out) return;
  if (a.epi == EPI_F32) {
    a.out[slot * a.slot_stride + static_cast<long long>(m) * a.ld_out + j] = acc;
    return;
  }
  float v = acc;
  if (a.epi == EPI_GELU_BF16) v = gelu_erf(acc);
  if (swiglu) v = silu(acc) * accu;
  const long long shard = j / a.shard_cols, lc = j % a.shard_cols;
  a.out[shard * a.shard_stride + static_cast<long long>(m) * a.ld_out + lc] = v;
}

// ---- decode activation ------------------------------------------------------

// h[s][t][j] for t < M, s < T, j < Fs (h is [T][M][Fs] bfloat16).
__global__ void decode_act_kernel(const float *P, int slots, long long slot_stride, long long ldp,
                                  int M, int T, int Fs, int act, int swiglu_rows,
                                  __nv_bfloat16 *h) {
  pdl_trigger();
  pdl_wait();  // the partials come from the GEMM before
  const long long total = static_cast<long long>(M) * T * Fs;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(e % Fs);
    const int t = static_cast<int>((e / Fs) % M);
    const int s = static_cast<int>(e / (static_cast<long long>(Fs) * M));
    long long grow;
    if (swiglu_rows)
      grow = static_cast<long long>(s) * 2 * Fs + (j / kSwigluGranule) * (2 * kSwigluGranule) +
             j % kSwigluGranule;
    else
      grow = static_cast<long long>(s) * Fs + j;
    const float *p = P + static_cast<long long>(t) * ldp + grow;
    float g = p[0];
    for (int sl = 1; sl < slots; ++sl) g += p[sl * slot_stride];
    float v;
    if (swiglu_rows) {
      float u = p[kSwigluGranule];
      for (int sl = 1; sl < slots; ++sl) u += p[sl * slot_stride + kSwigluGranule];
      v = silu(g) * u;
    } else {
      v = (act == TP_ACT_GELU_ERF) ? gelu_erf(g) : g;
    }
    h[e] = __float2bfloat16_rn(v);
  }
}

// Launch as a programmatic dependent of the previous kernel on the stream (the kernel calls
// pdl_wait before reading anything).
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), int grid, int threads, cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

int grid_for(long long items, int threads, int num_sms, int per_sm) {
  long long g = (items + threads - 1) / threads;
  const long long cap = static_cast<long long>(num_sms) * per_sm;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_shard_sum(const float *const *parts, int T, long long n, float *Z, int num_sms,
                             cudaStream_t stream) {
  if (T < 1 || T > kMaxParts) return cudaErrorInvalidValue;
  if (n <= 0) return cudaSuccess;
  PartList L{};
  bool aligned = (reinterpret_cast<uintptr_t>(Z) & 15u) == 0;
  for (int t = 0; t < T; ++t) {
    L.p[t] = parts[t];
    aligned = aligned && ((reinterpret_cast<uintptr_t>(parts[t]) & 15u) == 0);
  }
  constexpr int threads = 256;
  long long n4 = aligned ? n / 4 : 0;
  if (n4 > 0) {
    const int grid = grid_for(n4, threads, num_sms, 8);
    cudaError_t e;
    switch (T) {
      case 1: e = launch_dependent(shard_sum_fixed<1>, grid, threads, stream, L, n4, Z); break;
      case 2: e = launch_dependent(shard_sum_fixed<2>, grid, threads, stream, L, n4, Z); break;
      case 4: e = launch_dependent(shard_sum_fixed<4>, grid, threads, stream, L, n4, Z); break;
      case 8: e = launch_dependent(shard_sum_fixed<8>, grid, threads, stream, L, n4, Z); break;
      case 16: e = launch_dependent(shard_sum_fixed<16>, grid, threads, stream, L, n4, Z); break;
      default: e = launch_dependent(shard_sum_any, grid, threads, stream, L, T, n4, Z); break;
    }
    if (e != cudaSuccess) return e;
  }
  const long long first = n4 * 4;
  if (first < n) {
    const int grid = grid_for(n - first, threads, num_sms, 8);
    return launch_dependent(shard_sum_scalar, grid, threads, stream, L, T, first, n, Z);
  }
  return cudaSuccess;
}

cudaError_t launch_shard_sum_strided(const float *P, int slots, long long slot_stride, long long n,
                                     float *Z, int num_sms, cudaStream_t stream) {
  if (slots < 1 || slots > kMaxParts) return cudaErrorInvalidValue;
  const float *parts[kMaxParts];
  for (int s = 0; s < slots; ++s) parts[s] = P + s * slot_stride;
  return launch_shard_sum(parts, slots, n, Z, num_sms, stream);
}

cudaError_t launch_reduce_scatter(const float *const *parts, int T, long long n, float *const *out,
                                  int num_sms, cudaStream_t stream) {
  if (T < 1 || T > kMaxParts || n % T != 0) return cudaErrorInvalidValue;
  if (n <= 0) return cudaSuccess;
  PartList L{};
  OutList O{};
  const long long nb = n / T;
  bool vec = nb % 4 == 0;
  for (int t = 0; t < T; ++t) {
    L.p[t] = parts[t];
    O.p[t] = out[t];
    vec = vec && ((reinterpret_cast<uintptr_t>(parts[t]) | reinterpret_cast<uintptr_t>(out[t])) & 15u) == 0;
  }
  constexpr int threads = 256;
  if (vec) {
    reduce_scatter_vec<<<grid_for(n / 4, threads, num_sms, 8), threads, 0, stream>>>(L, T, O, nb / 4,
                                                                                    n / 4);
  } else {
    reduce_scatter_scalar<<<grid_for(n, threads, num_sms, 8), threads, 0, stream>>>(L, T, O, nb, n);
  }
  return cudaGetLastError();
}

cudaError_t launch_all_gather(const void *const *parts, int T, long long nb_bytes, void *out,
                              int num_sms, cudaStream_t stream) {
  if (T < 1 || T > kMaxParts || nb_bytes < 0) return cudaErrorInvalidValue;
  if (nb_bytes == 0) return cudaSuccess;
  ConstList L{};
  bool vec = nb_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
  for (int t = 0; t < T; ++t) {
    L.p[t] = static_cast<const uint8_t *>(parts[t]);
    vec = vec && (reinterpret_cast<uintptr_t>(parts[t]) & 15u) == 0;
  }
  constexpr int threads = 256;
  if (vec)
    all_gather_vec<<<grid_for(nb_bytes / 16 * T, threads, num_sms, 8), threads, 0, stream>>>(
        L, T, nb_bytes / 16, static_cast<uint4 *>(out));
  else
    all_gather_bytes<<<grid_for(nb_bytes * T, threads, num_sms, 8), threads, 0, stream>>>(
        L, T, nb_bytes, static_cast<uint8_t *>(out));
  return cudaGetLastError();
}

cudaError_t launch_shard_sum_bf16(const float *const *parts, int T, long long n, void *Z, int num_sms,
                                  cudaStream_t stream) {
  if (T < 1 || T > kMaxParts) return cudaErrorInvalidValue;
  if (n <= 0) return cudaSuccess;
  PartList L{};
  bool aligned = (reinterpret_cast<uintptr_t>(Z) & 7u) == 0;
  for (int t = 0; t < T; ++t) {
    L.p[t] = parts[t];
    aligned = aligned && ((reinterpret_cast<uintptr_t>(parts[t]) & 15u) == 0);
  }
  constexpr int threads = 256;
  const long long n4 = aligned ? n / 4 : 0;
  __nv_bfloat16 *z = static_cast<__nv_bfloat16 *>(Z);
  if (n4 > 0)
    shard_sum_bf16_vec<<<grid_for(n4, threads, num_sms, 8), threads, 0, stream>>>(L, T, n4, z);
  if (n4 * 4 < n)
    shard_sum_bf16_scalar<<<grid_for(n - n4 * 4, threads, num_sms, 8), threads, 0, stream>>>(
        L, T, n4 * 4, n, z);
  return cudaGetLastError();
}

cudaError_t launch_residual(const void *x, const float *z, float *h, void *hb, long long n, int num_sms,
                            cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  residual_kernel<<<grid_for(n, 256, num_sms, 8), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16 *>(x), z, h, static_cast<__nv_bfloat16 *>(hb), n);
  return cudaGetLastError();
}

cudaError_t launch_add_inplace(float *out, const float *h, long long n, int num_sms, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  add_inplace_kernel<<<grid_for(n, 256, num_sms, 8), 256, 0, stream>>>(out, h, n);
  return cudaGetLastError();
}

cudaError_t launch_pack(PackMode mode, const void *src, long long src_ld, void *dst, int S, long long R,
                        long long K, int esize, long long F, long long H, long long W,
                        cudaStream_t stream) {
  if (S < 1 || R < 1 || K < 1) return cudaErrorInvalidValue;
  if (esize == 2 && K % 64 != 0) return cudaErrorInvalidValue;  // whole k-tiles only
  const long long gy = (R + 31) / 32, gx = (K + 31) / 32;
  if (gy > 65535 || gx > 2147483647LL || S > 65535) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy), static_cast<unsigned>(S));
  dim3 block(32, 8);
  if (esize == 2)
    pack_kernel<uint16_t><<<grid, block, 0, stream>>>(mode, true, static_cast<const uint16_t *>(src), src_ld,
                                                      static_cast<uint16_t *>(dst), R, K, F, H, W);
  else if (esize == 4)
    pack_kernel<uint32_t><<<grid, block, 0, stream>>>(mode, false, static_cast<const uint32_t *>(src), src_ld,
                                                      static_cast<uint32_t *>(dst), R, K, F, H, W);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_unpack(PackMode mode, const void *packed, void *dst, int s, int S, int which,
                          long long R, long long K, int esize, long long W, cudaStream_t stream) {
  const int grid = 1024, threads = 256;
  if (esize == 2)
    unpack_kernel<uint16_t><<<grid, threads, 0, stream>>>(
        mode, true, static_cast<const uint16_t *>(packed), static_cast<uint16_t *>(dst), s, S, which, R, K, W);
  else if (esize == 4)
    unpack_kernel<uint32_t><<<grid, threads, 0, stream>>>(
        mode, false, static_cast<const uint32_t *>(packed), static_cast<uint32_t *>(dst), s, S, which, R, K, W);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_simt_gemm(const SimtArgs &a, cudaStream_t stream) {
  const int n_out = (a.epi == EPI_SWIGLU_BF16) ? a.N / 2 : a.N;
  const int slots = (a.nseg + a.segs_per_slot - 1) / a.segs_per_slot;
  if (a.M <= 0 || n_out <= 0) return cudaSuccess;
  dim3 grid((n_out + kSimtTile - 1) / kSimtTile, (a.M + kSimtTile - 1) / kSimtTile, slots);
  if (grid.y > 65535 || grid.z > 65535) return cudaErrorInvalidValue;
  simt_gemm_kernel<<<grid, dim3(kSimtTile, kSimtTile), 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode_act(const float *P, int slots, long long slot_stride, long long ldp, int M,
                              int T, int Fs, int act, bool swiglu_rows, void *h, cudaStream_t stream) {
  const long long total = static_cast<long long>(M) * T * Fs;
  if (total <= 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = grid_for(total, 256, sms, 8);
  return launch_dependent(decode_act_kernel, grid, 256, stream, P, slots, slot_stride, ldp, M, T, Fs, act,
                          swiglu_rows ? 1 : 0, static_cast<__nv_bfloat16 *>(h));
}

}  // namespace tp
