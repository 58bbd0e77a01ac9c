#pragma once
// tp_gemm_impl.cuh - the tensor-core GEMM of the tensor-parallel MLP on sm_103a
// (kernel templates; instantiated by tp_gemm.cu and tp_gemm_train.cu).
//
// One persistent, warp-specialised kernel serves every GEMM of the path:
//   - the column-parallel first layer Y_i = act(X W1_i) for all shards at
//     once, with GeLU / SwiGLU / identity fused into the epilogue and Y_i
//     stored as bfloat16 in shard i's own buffer ("Tensor Parallelism in
//     Action: Megatron-LM Matrix Splitting", section 1 "Column Parallel";
//     section 2, question 2, for why the activation stays local);
//   - the row-parallel second layer Z_i = Y_i W2_i, either as T float32
//     partials (one output slot per shard, summed afterwards by the
//     shard-sum kernel) or with one TMEM accumulator running over every
//     shard's K range, so that the all-reduce-sum happens inside the
//     accumulator ("Slice the matrix itself", section "Mathematical
//     formulation - row-parallel matrix multiplication summation");
//   - the memory-bound decode shapes with the operands swapped: the weight
//     rows are the 128-row MMA operand, the (<= 16) tokens the N = 16 one.
//
// Roles (192 threads): warp 0 issues TMA loads into a STAGES-deep ring of
// shared-memory tiles (128-byte swizzle); warp 1 allocates tensor memory and
// one of its threads issues tcgen05.mma (bf16 x bf16 -> fp32 in TMEM); warps
// 2..5 drain a finished accumulator (tcgen05.ld), apply the epilogue and
// store, while the MMA warp already fills the other accumulator.  Every wait
// is bounded (see tp_device.cuh): a wait that runs out sets the device
// status word and the CTA returns after letting its in-flight copies and
// MMAs finish and releasing its tensor memory.
#include <cuda_bf16.h>

#include <atomic>
#include <cstring>
#include <utility>

#include "tp_device.cuh"
#include "tp_internal.h"

namespace tp {
namespace gemm_impl {
namespace {

constexpr int BM = 128;          // MMA M (rows of A per tile)
constexpr int BK = 64;           // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;

template <int BN>
struct Traits;
template <>
struct Traits<256> {
  static constexpr int STAGES = 4;
};
template <>
struct Traits<128> {
  static constexpr int STAGES = 6;
};
template <>
struct Traits<16> {
  static constexpr int STAGES = 8;
};

constexpr int kAcc = 2;  // TMEM accumulators (double buffer)

template <int BN>
__host__ __device__ constexpr uint32_t tmem_cols() {
  return kAcc * BN <= 32 ? 32 : kAcc * BN <= 64 ? 64 : kAcc * BN <= 128 ? 128
         : kAcc * BN <= 256 ? 256 : 512;
}

template <int BN>
__host__ __device__ constexpr size_t smem_bytes() {
  return 1024 + static_cast<size_t>(Traits<BN>::STAGES) * (BM * BK * 2 + BN * BK * 2) + 256;
}

struct Unit {
  int slot, m, n, kt0, kt1;
};

// Unit u -> (slot, m-tile, n-tile, k range).  Inside a slot, tiles run in
// groups of `group_m` m-tiles with m fastest, so the CTAs working at the
// same time share B tiles (and A rows) through L2.
__device__ __forceinline__ Unit decode_unit(int u, const GemmArgs &g) {
  Unit r;
  const int per_slot = g.m_tiles * g.n_tiles;
  r.slot = u / per_slot;
  const int t = u - r.slot * per_slot;
  const int per_group = g.group_m * g.n_tiles;
  const int grp = t / per_group;
  const int first_m = grp * g.group_m;
  const int gm = min(g.group_m, g.m_tiles - first_m);
  const int in = t - grp * per_group;
  r.m = first_m + in % gm;
  r.n = in / gm;
  r.kt0 = r.slot * g.kt_per_slot;
  r.kt1 = min(g.kt_total, r.kt0 + g.kt_per_slot);
  // a unit outside the tile grid or an empty K range is a bug in the work split: report it and
  // turn the unit into an empty one on tile (0, 0)
  if (!TP_CHECK(r.slot < g.slots && r.m < g.m_tiles && r.n < g.n_tiles && r.kt0 < r.kt1, g.status)) {
    r.m = r.n = 0;
    r.kt1 = r.kt0;
  }
  return r;
}

// K coordinate and third tensor-map coordinate of the k-tiles of one unit,
// advanced one k-tile at a time (no division on the producer's path).  An
// operand in mode 0 is [1][rows][K] (flat K), mode 1 [segments][rows][K per
// segment].
struct KCursor {
  int k, z;         // current K element and third coordinate (segmented operands)
  int kflat;        // current K element of the virtual axis
  int seg_end;      // K element at which the current segment ends
  __device__ __forceinline__ void start(int kt0, const GemmArgs &g) {
    z = kt0 / g.kt_per_seg;
    k = (kt0 - z * g.kt_per_seg) * BK;
    kflat = kt0 * BK;
    seg_end = g.kt_per_seg * BK;
  }
  __device__ __forceinline__ void next() {
    kflat += BK;
    k += BK;
    if (k == seg_end) {
      k = 0;
      ++z;
    }
  }
  __device__ __forceinline__ void coords(int mode, int &kc, int &zc) const {
    kc = mode == 1 ? k : mode == kKtileBlocked ? 0 : kflat;
    zc = mode == 1 ? z : mode == kKtileBlocked ? kflat / BK : 0;
  }
};

// Tensor-map coordinates (x, z) of the 64-row blocks [row0 + 64 i, row0 + 64 i + 64) of an
// MN-major operand tile (EPI_F32_MN): x is the row within its MN segment of `seg` rows, z the
// segment (seg = 0: one segment).  Set once per unit; a block never straddles segments.
template <int N>
struct MnBlocks {
  int x[N], z[N];
  __device__ __forceinline__ void set(int row0, int seg) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int r = row0 + 64 * i;
      z[i] = seg > 0 ? r / seg : 0;
      x[i] = r - z[i] * seg;
    }
  }
};
constexpr uint32_t kMnBlockBytes = 64 * BK * 2;  // one 64 x 64 box

// GeLU(x) = x/2 (1 + erf(x / sqrt 2)), erf by Abramowitz and Stegun, "Handbook of
// Mathematical Functions", formula 7.1.26: for u >= 0, erf(u) = 1 - (a1 t + a2 t^2 + a3 t^3 +
// a4 t^4 + a5 t^5) e^(-u^2), t = 1 / (1 + p u), |error| <= 1.5e-7 (the tensor-core path rounds
// the result to bfloat16, 2^-9 relative); erf(-u) = -erf(u).  Two MUFU operations and a few
// FMA-pipe ones per value, about half the library erff: the epilogue warps share their SM
// sub-partitions with the copy-issuing and MMA-issuing threads, so their arithmetic slows the
// main loop.
namespace as7126 {
constexpr float kP = 0.3275911f, kA1 = 0.254829592f, kA2 = -0.284496736f, kA3 = 1.421413741f,
                kA4 = -1.453152027f, kA5 = 1.061405429f;
constexpr float kRsqrt2 = 0.70710678118654752f, kNegLog2e = -1.4426950408889634f;
__device__ __forceinline__ float rcp(float d) {
  float t;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(d));
  return t;
}
}  // namespace as7126

// Two values at a time, with paired float32 operations.
__device__ __forceinline__ float2 gelu_erf2(float2 x) {
  using namespace as7126;
  const float2 u = __fmul2_rn(x, make_float2(kRsqrt2, kRsqrt2));
  const float2 au = make_float2(fabsf(u.x), fabsf(u.y));
  const float2 d = __ffma2_rn(make_float2(kP, kP), au, make_float2(1.0f, 1.0f));
  const float2 t = make_float2(rcp(d.x), rcp(d.y));
  float2 p = __ffma2_rn(t, make_float2(kA5, kA5), make_float2(kA4, kA4));
  p = __ffma2_rn(t, p, make_float2(kA3, kA3));
  p = __ffma2_rn(t, p, make_float2(kA2, kA2));
  p = __ffma2_rn(t, p, make_float2(kA1, kA1));
  p = __fmul2_rn(p, t);
  const float2 a = __fmul2_rn(__fmul2_rn(au, au), make_float2(kNegLog2e, kNegLog2e));
  const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
  const float2 q = __ffma2_rn(p, e, make_float2(-1.0f, -1.0f));
  const float2 h = __fmul2_rn(x, make_float2(0.5f, 0.5f));
  return __ffma2_rn(h, make_float2(copysignf(fabsf(q.x), u.x), copysignf(fabsf(q.y), u.y)), h);
}

// SiLU(g) = g / (1 + e^-g) with the ex2 and rcp approximations (relative error about 1e-7,
// far below bfloat16's); silu2 pairs the multiplications and rounds alike.
__device__ __forceinline__ float silu(float g) {
  return g * as7126::rcp(1.0f + ex2_approx(g * as7126::kNegLog2e));
}

__device__ __forceinline__ float2 silu2(float2 g) {
  const float2 a = __fmul2_rn(g, make_float2(as7126::kNegLog2e, as7126::kNegLog2e));
  const float2 r = make_float2(as7126::rcp(1.0f + ex2_approx(a.x)), as7126::rcp(1.0f + ex2_approx(a.y)));
  return __fmul2_rn(g, r);
}

// GeLU'(y) = Phi(y) + y phi(y), Phi(y) = (1 + erf(y / sqrt 2)) / 2, phi(y) = e^(-y^2 / 2) /
// sqrt(2 pi); erf by the same formula 7.1.26 as gelu_erf2.  With u = y / sqrt 2 the formula's
// e^(-u^2) is e^(-y^2 / 2), so one exponential serves both terms: for u >= 0, Phi(y) = 1 - c and
// for u < 0, Phi(y) = c, where c = (a1 t + ... + a5 t^5) e^(-u^2) / 2 (the coefficients halved,
// which is exact).  Two values at a time with paired float32 operations.
namespace as7126 {
constexpr float kH1 = 0.5f * kA1, kH2 = 0.5f * kA2, kH3 = 0.5f * kA3, kH4 = 0.5f * kA4, kH5 = 0.5f * kA5;
constexpr float kInvSqrt2Pi = 0.39894228040143268f;
}  // namespace as7126

__device__ __forceinline__ float2 gelu_grad2(float2 y) {
  using namespace as7126;
  const float2 u = __fmul2_rn(y, make_float2(kRsqrt2, kRsqrt2));
  const float2 au = make_float2(fabsf(u.x), fabsf(u.y));
  const float2 d = __ffma2_rn(make_float2(kP, kP), au, make_float2(1.0f, 1.0f));
  const float2 t = make_float2(rcp(d.x), rcp(d.y));
  float2 p = __ffma2_rn(t, make_float2(kH5, kH5), make_float2(kH4, kH4));
  p = __ffma2_rn(t, p, make_float2(kH3, kH3));
  p = __ffma2_rn(t, p, make_float2(kH2, kH2));
  p = __ffma2_rn(t, p, make_float2(kH1, kH1));
  p = __fmul2_rn(p, t);
  const float2 a = __fmul2_rn(__fmul2_rn(au, au), make_float2(kNegLog2e, kNegLog2e));
  const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
  const float2 c = __fmul2_rn(p, e);
  const float2 phi_cdf = make_float2(u.x >= 0.0f ? 1.0f - c.x : c.x, u.y >= 0.0f ? 1.0f - c.y : c.y);
  return __ffma2_rn(__fmul2_rn(y, make_float2(kInvSqrt2Pi, kInvSqrt2Pi)), e, phi_cdf);
}

// s = sigmoid(g) = 1 / (1 + e^-g) for two values, by the ex2 and rcp approximations; the
// SwiGLU backward takes SiLU(g) = g s and SiLU'(g) = s (1 + g (1 - s)) from it.
__device__ __forceinline__ float2 sigmoid2(float2 g) {
  const float2 a = __fmul2_rn(g, make_float2(as7126::kNegLog2e, as7126::kNegLog2e));
  return make_float2(as7126::rcp(1.0f + ex2_approx(a.x)), as7126::rcp(1.0f + ex2_approx(a.y)));
}

// 32-byte global accesses: one instruction moves a whole 32-byte sector, where
// two 16-byte ones would each send half a sector (twice the requests and, for
// stores, twice the bytes through the crossbar).  The address must be 32-byte
// aligned.
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t *v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]), "r"(v[1]), "r"(v[2]),
               "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__device__ __forceinline__ void ld_global_v8(const void *p, uint32_t *v) {
  asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "l"(p)
               : "memory");
}

__device__ __forceinline__ bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// 32 consecutive bf16 (16-byte aligned) -> float; two 32-byte loads where the
// address allows.
__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16 *src, float (&v)[32]) {
  uint32_t w[16];
  if (aligned32(src)) {
    ld_global_v8(src, w);
    ld_global_v8(src + 16, w + 8);
  } else {
    const uint4 *p = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 q = p[j];
      w[4 * j] = q.x;
      w[4 * j + 1] = q.y;
      w[4 * j + 2] = q.z;
      w[4 * j + 3] = q.w;
    }
  }
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    v[2 * k] = __uint_as_float(w[k] << 16);
    v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// 32 float32 values of one row -> activation -> 32 bf16 at dst (16 B aligned;
// two 32-byte stores where the address allows).
template <int EPI>
__device__ __forceinline__ void store_act32(__nv_bfloat16 *dst, const uint32_t (&r)[32]) {
  uint32_t p[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float2 v = make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
    if (EPI == EPI_GELU_BF16) v = gelu_erf2(v);
    p[j] = pack_bf16x2(v.x, v.y);
  }
  if (aligned32(dst)) {
    st_global_v8(dst, p);
    st_global_v8(dst + 16, p + 8);
  } else {
    uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int j = 0; j < 4; ++j) d[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
  }
}

// Float32 output with the residual of a row-parallel layer (EPI_F32_RESID): `ncols` columns (a
// multiple of 32) of one accumulator, output row `row` (this thread's TMEM lane), columns
// n0 .. : out = acc (+ float32 residual aux) (+ bf16 residual aux2), and with out2 its bf16.
__device__ __forceinline__ void epilogue_resid_cols(uint32_t tb, int row, long long n0, int ncols,
                                                    const GemmArgs &g) {
  const bool valid = row < g.rows_valid;
  const long long off = static_cast<long long>(row) * g.ld_out + n0;
  float *out = static_cast<float *>(g.out) + off;
  const float *addf = static_cast<const float *>(g.aux);
  const __nv_bfloat16 *addb = static_cast<const __nv_bfloat16 *>(g.aux2);
  __nv_bfloat16 *outb = static_cast<__nv_bfloat16 *>(g.out2);
  // the float32 rows (output and residual) move 32 bytes at a time when aligned
  const bool wide = aligned32(out) && (!addf || aligned32(addf + off));
#pragma unroll 1
  for (int c = 0; c < ncols / 32; ++c) {
    uint32_t r[32];
    tmem_ld32(tb + c * 32, r);
    tmem_ld_wait();
    if (!valid) continue;
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    if (addf && wide) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t x[8];
        ld_global_v8(addf + off + c * 32 + 8 * j, x);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[8 * j + k] += __uint_as_float(x[k]);
      }
    } else if (addf) {
      const float4 *a = reinterpret_cast<const float4 *>(addf + off + c * 32);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 x = a[j];
        v[4 * j] += x.x;
        v[4 * j + 1] += x.y;
        v[4 * j + 2] += x.z;
        v[4 * j + 3] += x.w;
      }
    }
    if (addb) {
      const uint4 *a = reinterpret_cast<const uint4 *>(addb + off + c * 32);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 x = a[j];
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          v[8 * j + 2 * k] += __uint_as_float(w[k] << 16);
          v[8 * j + 2 * k + 1] += __uint_as_float(w[k] & 0xFFFF0000u);
        }
      }
    }
    if (wide) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t x[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = __float_as_uint(v[8 * j + k]);
        st_global_v8(out + c * 32 + 8 * j, x);
      }
    } else {
      float4 *d = reinterpret_cast<float4 *>(out + c * 32);
#pragma unroll
      for (int j = 0; j < 8; ++j) d[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
    if (outb) {
      uint32_t vb[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) vb[j] = __float_as_uint(v[j]);
      store_act32<EPI_IDENT_BF16>(outb + off + c * 32, vb);
    }
  }
}

// Epilogue of one tile by the 128 epilogue threads: each thread owns TMEM
// lane `row_in_tile`, i.e. output row row0 + row_in_tile; `tb` addresses that
// lane's quarter at the accumulator's first column.
template <int BN, int EPI>
__device__ __forceinline__ void epilogue_tile(uint32_t tb, const Unit &t, int row0, int row_in_tile,
                                              const GemmArgs &g) {
  if constexpr (EPI == EPI_F32_T) {
    static_assert(BN == 16, "swapped epilogue is the N = 16 decode tile");
    uint32_t r[16];
    tmem_ld16(tb, r);
    tmem_ld_wait();
    const int feat = row0 + row_in_tile;
    if (feat < g.rows_valid) {
      float *out = static_cast<float *>(g.out) + t.slot * g.slot_stride + feat;
#pragma unroll
      for (int j = 0; j < BN; ++j)
        if (j < g.cols_valid) out[j * g.ld_out] = __uint_as_float(r[j]);
    }
  } else if constexpr (EPI == EPI_F32 || EPI == EPI_F32_MN) {
    const int row = row0 + row_in_tile;
    const bool valid = row < g.rows_valid;
    float *out = static_cast<float *>(g.out) + t.slot * g.slot_stride +
                 static_cast<long long>(row) * g.ld_out + static_cast<long long>(t.n) * BN;
    const bool wide = aligned32(out);  // rows of a multiple of 8 floats on a 32-byte base
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tb + c * 32, r);
      tmem_ld_wait();
      if (valid && wide) {
#pragma unroll
        for (int j = 0; j < 4; ++j) st_global_v8(out + c * 32 + 8 * j, r + 8 * j);
      } else if (valid) {
        float4 *d = reinterpret_cast<float4 *>(out + c * 32);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          d[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                             __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
      }
    }
  } else if constexpr (EPI == EPI_F32_RESID) {
    epilogue_resid_cols(tb, row0 + row_in_tile, t.n * BN, BN, g);
  } else if constexpr (EPI == EPI_SWIGLU_BF16) {
    constexpr int HALF = BN / 2;
    const int row = row0 + row_in_tile;
    const bool valid = row < g.rows_valid;
    const long long col0 = static_cast<long long>(t.n) * HALF;
    const long long shard = col0 / g.shard_cols;
    const long long lc = col0 - shard * g.shard_cols;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(g.out) + shard * g.shard_stride +
                         static_cast<long long>(row) * g.ld_out + lc;
#pragma unroll 1
    for (int c = 0; c < HALF / 32; ++c) {
      uint32_t gr[32], ur[32];
      tmem_ld32(tb + c * 32, gr);
      tmem_ld32(tb + HALF + c * 32, ur);
      tmem_ld_wait();
      if (valid) {
        uint32_t h[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          h[j] = __float_as_uint(silu(__uint_as_float(gr[j])) * __uint_as_float(ur[j]));
        store_act32<EPI_IDENT_BF16>(out + c * 32, h);
      }
    }
  } else if constexpr (EPI == EPI_SWIGLU_SAVE_BF16) {
    constexpr int HALF = BN / 2;
    const int row = row0 + row_in_tile;
    const bool valid = row < g.rows_valid;
    const long long col0 = static_cast<long long>(t.n) * HALF;
    const long long shard = col0 / g.shard_cols;
    const long long off = shard * g.shard_stride + static_cast<long long>(row) * g.ld_out +
                          (col0 - shard * g.shard_cols);
#pragma unroll 1
    for (int c = 0; c < HALF / 32; ++c) {
      uint32_t gr[32], ur[32];
      tmem_ld32(tb + c * 32, gr);
      tmem_ld32(tb + HALF + c * 32, ur);
      tmem_ld_wait();
      if (valid) {
        uint32_t h[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          h[j] = __float_as_uint(silu(__uint_as_float(gr[j])) * __uint_as_float(ur[j]));
        store_act32<EPI_IDENT_BF16>(static_cast<__nv_bfloat16 *>(g.out) + off + c * 32, h);
        store_act32<EPI_IDENT_BF16>(static_cast<__nv_bfloat16 *>(g.out2) + off + c * 32, gr);
        store_act32<EPI_IDENT_BF16>(static_cast<__nv_bfloat16 *>(g.out3) + off + c * 32, ur);
      }
    }
  } else if constexpr (EPI == EPI_GELU_SAVE_BF16 || EPI == EPI_DGELU_BF16 ||
                       EPI == EPI_DSWIGLU_BF16) {
    const int row = row0 + row_in_tile;
    const bool valid = row < g.rows_valid;
    const long long col0 = static_cast<long long>(t.n) * BN;
    const long long shard = col0 / g.shard_cols;
    const long long off = shard * g.shard_stride + static_cast<long long>(row) * g.ld_out +
                          (col0 - shard * g.shard_cols);
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tb + c * 32, r);
      tmem_ld_wait();
      if (!valid) continue;
      __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(g.out) + off + c * 32;
      if constexpr (EPI == EPI_GELU_SAVE_BF16) {
        store_act32<EPI_GELU_BF16>(out, r);
        store_act32<EPI_IDENT_BF16>(static_cast<__nv_bfloat16 *>(g.out2) + off + c * 32, r);
      } else if constexpr (EPI == EPI_DGELU_BF16) {
        float p[32];
        load_bf16x32(static_cast<const __nv_bfloat16 *>(g.aux) + off + c * 32, p);
        uint32_t d[32];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 gd = __fmul2_rn(make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])),
                                       gelu_grad2(make_float2(p[2 * j], p[2 * j + 1])));
          d[2 * j] = __float_as_uint(gd.x);
          d[2 * j + 1] = __float_as_uint(gd.y);
        }
        store_act32<EPI_IDENT_BF16>(out, d);
      } else {
        float gv[32], uv[32];
        load_bf16x32(static_cast<const __nv_bfloat16 *>(g.aux) + off + c * 32, gv);
        load_bf16x32(static_cast<const __nv_bfloat16 *>(g.aux2) + off + c * 32, uv);
        uint32_t dg[32], du[32];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 dh = make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
          const float2 g2 = make_float2(gv[2 * j], gv[2 * j + 1]), u2 = make_float2(uv[2 * j], uv[2 * j + 1]);
          const float2 sg = sigmoid2(g2);
          // dg = dh u SiLU'(g), SiLU'(g) = s (1 + g (1 - s));  du = dh SiLU(g) = dh g s
          const float2 one = make_float2(1.0f, 1.0f);
          const float2 d1 = __ffma2_rn(g2, __ffma2_rn(sg, make_float2(-1.0f, -1.0f), one), one);
          const float2 a = __fmul2_rn(__fmul2_rn(dh, u2), __fmul2_rn(sg, d1));
          const float2 b = __fmul2_rn(dh, __fmul2_rn(g2, sg));
          dg[2 * j] = __float_as_uint(a.x);
          dg[2 * j + 1] = __float_as_uint(a.y);
          du[2 * j] = __float_as_uint(b.x);
          du[2 * j + 1] = __float_as_uint(b.y);
        }
        store_act32<EPI_IDENT_BF16>(out, dg);
        store_act32<EPI_IDENT_BF16>(static_cast<__nv_bfloat16 *>(g.out2) + off + c * 32, du);
      }
    }
  } else if constexpr (EPI == EPI_QKV_HEADS_BF16) {
    // global column -> (shard, Q/K/V, head, dim); 32-column chunks stay in one head
    const int row = row0 + row_in_tile;
    const bool valid = row < g.rows_valid;
    const long long W = g.shard_cols / 3;
    const long long hps = W / g.head_dim;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tb + c * 32, r);
      tmem_ld_wait();
      if (!valid) continue;
      const long long gc = static_cast<long long>(t.n) * BN + c * 32;
      const long long sh = gc / g.shard_cols, lc = gc - sh * g.shard_cols;
      const long long part = lc / W, within = lc - part * W;
      const long long head = sh * hps + within / g.head_dim, dim = within % g.head_dim;
      const long long block = part * g.n_heads + head;
      store_act32<EPI_IDENT_BF16>(static_cast<__nv_bfloat16 *>(g.out) +
                                      (block * g.rows_valid + row) * g.head_dim + dim, r);
    }
  } else {  // EPI_GELU_BF16, EPI_IDENT_BF16
    const int row = row0 + row_in_tile;
    const bool valid = row < g.rows_valid;
    const long long col0 = static_cast<long long>(t.n) * BN;
    const long long shard = col0 / g.shard_cols;
    const long long lc = col0 - shard * g.shard_cols;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(g.out) + shard * g.shard_stride +
                         static_cast<long long>(row) * g.ld_out + lc;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tb + c * 32, r);
      tmem_ld_wait();
      if (valid) store_act32<EPI>(out + c * 32, r);
    }
  }
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    tp_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                   const GemmArgs g) {
  constexpr int STAGES = Traits<BN>::STAGES;
  constexpr uint32_t A_BYTES = BM * BK * 2;
  constexpr uint32_t B_BYTES = BN * BK * 2;
  constexpr uint32_t TMEM_COLS = tmem_cols<BN>();
  constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + STAGES * A_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sB + STAGES * B_BYTES);
  // barriers: full[STAGES] | empty[STAGES] | tfull[kAcc] | tempty[kAcc] | drain | never
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 2 * kAcc + 2);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + kAcc + a); };
  const uint32_t drain = bar0 + 8u * (2 * STAGES + 2 * kAcc);
  const uint32_t never = drain + 8u;  // nothing ever arrives here (timeout test)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < kAcc; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), kEpiThreads);
    }
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&mapA);
    prefetch_tmap(&mapB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the set-up above overlaps the previous kernel's tail; its outputs are read only from here on
  pdl_trigger();
  pdl_wait();

  const WaitCtl w{abort_flag, g.status, g.wait_limit_ns};
  const int units = g.slots * g.m_tiles * g.n_tiles;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer ----
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      constexpr bool amn = EPI == EPI_F32_MN, bmn = EPI == EPI_F32_MN;
      constexpr int kBBlocks = BN >= 64 ? BN / 64 : 1;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit t = decode_unit(u, g);
        MnBlocks<BM / 64> ablk;
        MnBlocks<kBBlocks> bblk;
        if constexpr (amn) ablk.set(t.m * BM, g.a_mn_seg);
        if constexpr (bmn) bblk.set(t.n * BN, g.b_mn_seg);
        KCursor kc;
        kc.start(t.kt0, g);
        for (int kt = t.kt0; kt < t.kt1; ++kt, kc.next()) {
          if (!wait_bar_spin(empty_bar(stage), phase ^ 1u, w)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES);
          int ak, az, bk, bz;
          kc.coords(g.a_seg, ak, az);
          kc.coords(g.b_seg, bk, bz);
          if constexpr (amn) {
            // two 64-row MN blocks per copy (kMnPairBox)
#pragma unroll
            for (int i = 0; i < BM / 64; i += kMnPairBox)
              tma_load_4d(smem_u32(sA + stage * A_BYTES + i * kMnBlockBytes), &mapA, fb, 0, kc.kflat,
                          ablk.x[i] / 64, ablk.z[i]);
          } else {
            tma_load_3d(smem_u32(sA + stage * A_BYTES), &mapA, fb, ak, t.m * BM, az);
          }
          if constexpr (bmn && BN >= 128) {
#pragma unroll
            for (int i = 0; i < kBBlocks; i += kMnPairBox)
              tma_load_4d(smem_u32(sB + stage * B_BYTES + i * kMnBlockBytes), &mapB, fb, 0, kc.kflat,
                          bblk.x[i] / 64, bblk.z[i]);
          } else {
            tma_load_3d(smem_u32(sB + stage * B_BYTES), &mapB, fb, bk, t.n * BN, bz);
          }
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Every copy already issued must land before the CTA may exit.
        for (int s = 0; s < STAGES; ++s)
          if ((issued >> s) & 1u) drain_bar(full_bar(s), (last_par >> s) & 1u, g.status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer ----
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      // Under a test wait limit, first wait for an event that never happens,
      // so that the timeout path runs with copies in flight.
      bool ok = !(g.wait_limit_ns < kShortLimitNs) || wait_bar(never, 0u, w);
      constexpr bool amn = EPI == EPI_F32_MN, bmn = EPI == EPI_F32_MN;
      constexpr uint32_t idesc = IDESC | (amn ? kIdescMnA : 0u) | (bmn ? kIdescMnB : 0u);
      // one K = 16 step: +32 B (K-major) or +2 KiB (MN-major), in 16-byte units
      constexpr uint32_t astep = amn ? 128u : 2u, bstep = bmn ? 128u : 2u;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit t = decode_unit(u, g);
        if (!wait_bar_spin(tempty_bar(acc), acc_phase ^ 1u, w)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kt = t.kt0; kt < t.kt1; ++kt) {
          if (!wait_bar_spin(full_bar(stage), phase, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(sA + stage * A_BYTES), sb = smem_u32(sB + stage * B_BYTES);
          const uint64_t ad = amn ? sw128_mnmajor_desc(sa) : sw128_kmajor_desc(sa);
          const uint64_t bd = bmn ? sw128_mnmajor_desc(sb) : sw128_kmajor_desc(sb);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma_bf16(d, ad + astep * k, bd + bstep * k, idesc, (kt > t.kt0 || k > 0) ? 1u : 0u);
          tc_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(tfull_bar(acc));
        if (++acc == kAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // Every MMA issued must be complete before tensor memory is released.
      tc_commit(drain);
      drain_bar(drain, 0u, g.status);
    }
    __syncwarp();
  } else {
    // ---- epilogue (warps 2..5) ----
    const int q = warp & 3;  // TMEM lanes [32q, 32q + 32) are this warp's
    const int row_in_tile = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const Unit t = decode_unit(u, g);
      const bool ok = wait_bar(tfull_bar(acc), acc_phase, w);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(acc * BN);
      epilogue_tile<BN, EPI>(tb, t, t.m * BM, row_in_tile, g);
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
      if (++acc == kAcc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---- CTA-pair variant ------------------------------------------------------
//
// Cluster of 2 CTAs on a 256 x 256 output tile.  CTA r loads rows
// [128 r, 128 r + 128) of the A tile and rows [128 r, 128 r + 128) of the B
// tile into its own shared memory (32 KiB per stage); both CTAs' copies
// complete on CTA 0's stage barrier, which CTA 0 arms for both halves.  One
// thread of CTA 0 issues tcgen05.mma.cta_group::2 (M = 256, N = 256), which
// reads both CTAs' tiles and leaves rows [128 r, 128 r + 128) x 256 columns
// in CTA r's tensor memory.  Commits are multicast to both CTAs' barriers;
// the epilogue warps of both CTAs release an accumulator on CTA 0's barrier.
// On an abort CTA 0 waits for the stages it armed; CTA 1, whose copies
// complete on CTA 0's barriers, waits a bounded time for its copies in flight.
#ifndef TP_PAIR_STAGES
#define TP_PAIR_STAGES 7
#endif
constexpr int kPairStages = TP_PAIR_STAGES;
// Time CTA 1 leaves its in-flight copies to land after an abort.
constexpr unsigned long long kPeerDrainNs = 200000ull;
constexpr int kPairBN = 256;

// Epilogues that leave through TMA stores: each epilogue warp stages 32 rows x 128 bytes of its
// output in shared memory (two buffers) and one lane stores them as a box, instead of each
// thread writing its row with 16-byte stores (32 rows per store instruction).  The epilogue
// runs while the next tile's main loop does, so every instruction it saves helps that loop.
// The staging space (32 KiB) takes one stage of the ring.
template <int EPI>
__host__ __device__ constexpr bool tma_store_epi() {
  return EPI == EPI_GELU_BF16 || EPI == EPI_IDENT_BF16 || EPI == EPI_F32 || EPI == EPI_SWIGLU_BF16;
}
constexpr uint32_t kStoreBufBytes = 32 * 128;  // 32 rows x 128 B, 128-byte swizzle
// Stages of the ring; the wide schedule's stages hold up to kWideMaxN / 2 B rows per CTA.
template <int EPI, bool WIDE = false>
__host__ __device__ constexpr int pair_stages() {
  return WIDE ? 4 : tma_store_epi<EPI>() ? kPairStages - 1 : kPairStages;
}
template <bool WIDE = false>
__host__ __device__ constexpr uint32_t pair_b_bytes() {
  return static_cast<uint32_t>(WIDE ? kWideMaxN / 2 : kPairBN / 2) * BK * 2;
}
template <int EPI, bool WIDE = false>
__host__ __device__ constexpr size_t pair_smem_bytes() {
  return 1024 + static_cast<size_t>(pair_stages<EPI, WIDE>()) * (128 * BK * 2 + pair_b_bytes<WIDE>()) +
         (tma_store_epi<EPI>() ? 8 * kStoreBufBytes : 0) + 512;
}
static_assert(pair_smem_bytes<EPI_F32_RESID>() <= 232448, "pair kernel exceeds 227 KiB of shared memory");
static_assert(pair_smem_bytes<EPI_F32>() <= 232448, "pair kernel exceeds 227 KiB of shared memory");
static_assert(pair_smem_bytes<EPI_F32, true>() <= 232448, "wide pair kernel exceeds 227 KiB of shared memory");
static_assert(kWideMaxN > 256 && kWideMaxN <= 512 && kWideMaxN % 32 == 0, "wide tiles: two MMAs, one TMEM allocation");

// One cluster's work on the wide schedule (GemmArgs::wide_*): `width` columns from n0 of
// 256-row block m0.  The row blocks of one column range run side by side (they share its B
// tiles through L2).
struct WideUnit {
  int m0, n0, width;
};
__device__ __forceinline__ WideUnit decode_wide(int u, const GemmArgs &g) {
  WideUnit r;
  r.m0 = u % g.m_tiles;
  const int j = u / g.m_tiles;  // tile of the row block: wide_nb of wide_bn columns, then 32 fewer
  const int narrow = j - g.wide_nb;
  r.width = narrow < 0 ? g.wide_bn : g.wide_bn - 32;
  r.n0 = narrow < 0 ? j * g.wide_bn : g.wide_nb * g.wide_bn + narrow * (g.wide_bn - 32);
  // a tile outside the output or of a width the kernel cannot take is a bug in the plan:
  // report it and run the first tile instead
  if (!TP_CHECK(r.m0 < g.m_tiles && j < g.wide_q && r.width > 256 && r.width <= kWideMaxN &&
                    r.n0 + r.width <= g.cols_valid,
                g.status)) {
    r.m0 = 0;
    r.n0 = 0;
    r.width = g.wide_bn;
  }
  return r;
}

// Float32 epilogue of `ncols` columns (a multiple of 32) of one accumulator through the warp's
// staging buffers and TMA stores (output columns x0 ..; TMEM lanes = rows wrow .. wrow + 31).
__device__ __forceinline__ void epilogue_f32_cols(uint32_t tb, int x0, int ncols, int wrow, int lane,
                                                  const GemmArgs &g, const CUtensorMap *mapO, uint8_t *bufs,
                                                  uint32_t &nstore) {
  const bool rows_in = wrow < g.rows_valid;
#pragma unroll 1
  for (int c = 0; c < ncols / 32; ++c) {
    uint8_t *buf = bufs + (nstore & 1u) * kStoreBufBytes;
    if (lane == 0) bulk_wait_read<1>();  // the store that last read this buffer is done with it
    __syncwarp();
    uint32_t w[32];
    tmem_ld32(tb + c * 32, w);
    tmem_ld_wait();
    tmem_reg_fence(w);
    uint4 *row = reinterpret_cast<uint4 *>(buf + lane * 128);
#pragma unroll
    for (int j = 0; j < 8; ++j) row[j ^ (lane & 7)] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (rows_in) tma_store_3d(mapO, smem_u32(buf), x0 + c * 32, wrow, 0);
      bulk_commit();
    }
    ++nstore;
  }
}

// Epilogue of one 256-column accumulator by one warp through TMA stores: TMEM lanes
// [32 q, 32 q + 32) are output rows wrow .. wrow + 31; 128-byte column chunks (64 bf16 or 32
// float32) go through the warp's two staging buffers, row `lane` with its 16-byte pieces in
// the 128-byte swizzle.  mapO is [segments][rows][columns]: shards of the bf16 Y, or slots of
// the float32 output; rows past the map's row count are not stored.
template <int BN, int EPI>
__device__ __forceinline__ void epilogue_tile_tma(uint32_t tb, const Unit &t, int wrow, int lane, const GemmArgs &g,
                                                  const CUtensorMap *mapO, uint8_t *bufs, uint32_t &nstore) {
  constexpr bool f32 = EPI == EPI_F32;
  constexpr bool swiglu = EPI == EPI_SWIGLU_BF16;  // 128 gate then 128 up columns -> 128 outputs
  constexpr int CW = f32 ? 32 : 64;                 // output columns per 128-byte row chunk
  constexpr int OUT_COLS = swiglu ? BN / 2 : BN;
  int x0, z;
  if constexpr (f32) {
    x0 = t.n * BN;
    z = t.slot;
  } else {
    const int col0 = t.n * OUT_COLS;
    z = col0 / g.shard_cols;
    x0 = col0 - z * g.shard_cols;
  }
  const bool rows_in = wrow < g.rows_valid;
#pragma unroll 1
  for (int c = 0; c < OUT_COLS / CW; ++c) {
    uint8_t *buf = bufs + (nstore & 1u) * kStoreBufBytes;
    if (lane == 0) bulk_wait_read<1>();  // the store that last read this buffer is done with it
    __syncwarp();
    uint32_t w[32];
    if constexpr (f32) {
      tmem_ld32(tb + c * 32, w);
      tmem_ld_wait();
      tmem_reg_fence(w);
    } else if constexpr (swiglu) {
      uint32_t g0[32], g1[32], u0[32], u1[32];
      tmem_ld32(tb + c * 64, g0);
      tmem_ld32(tb + c * 64 + 32, g1);
      tmem_ld32(tb + BN / 2 + c * 64, u0);
      tmem_ld32(tb + BN / 2 + c * 64 + 32, u1);
      tmem_ld_wait();
      tmem_reg_fence(g0);
      tmem_reg_fence(g1);
      tmem_reg_fence(u0);
      tmem_reg_fence(u1);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float2 ha = __fmul2_rn(silu2(make_float2(__uint_as_float(g0[2 * j]), __uint_as_float(g0[2 * j + 1]))),
                                     make_float2(__uint_as_float(u0[2 * j]), __uint_as_float(u0[2 * j + 1])));
        const float2 hb = __fmul2_rn(silu2(make_float2(__uint_as_float(g1[2 * j]), __uint_as_float(g1[2 * j + 1]))),
                                     make_float2(__uint_as_float(u1[2 * j]), __uint_as_float(u1[2 * j + 1])));
        w[j] = pack_bf16x2(ha.x, ha.y);
        w[16 + j] = pack_bf16x2(hb.x, hb.y);
      }
    } else {
      uint32_t r0[32], r1[32];
      tmem_ld32(tb + c * 64, r0);
      tmem_ld32(tb + c * 64 + 32, r1);
      tmem_ld_wait();
      tmem_reg_fence(r0);
      tmem_reg_fence(r1);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float a0 = __uint_as_float(r0[2 * j]), a1 = __uint_as_float(r0[2 * j + 1]);
        float b0 = __uint_as_float(r1[2 * j]), b1 = __uint_as_float(r1[2 * j + 1]);
        if constexpr (EPI == EPI_GELU_BF16) {
          const float2 ga = gelu_erf2(make_float2(a0, a1)), gb = gelu_erf2(make_float2(b0, b1));
          a0 = ga.x;
          a1 = ga.y;
          b0 = gb.x;
          b1 = gb.y;
        }
        w[j] = pack_bf16x2(a0, a1);
        w[16 + j] = pack_bf16x2(b0, b1);
      }
    }
    uint4 *row = reinterpret_cast<uint4 *>(buf + lane * 128);
#pragma unroll
    for (int j = 0; j < 8; ++j) row[j ^ (lane & 7)] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (rows_in) tma_store_3d(mapO, smem_u32(buf), x0 + c * CW, wrow, z);
      bulk_commit();
    }
    ++nstore;
  }
}

// WIDE: the wide row-parallel schedule (EPI_F32 and EPI_F32_RESID): tiles of up to kWideMaxN
// columns, one per cluster at a time, as two MMAs per k-step (256 columns into TMEM columns 0 ..,
// the rest into 256 ..), each CTA loading its half of both B pieces (mapB: 128 rows; the second
// piece's half with mapB2 for the wide_bn-column tiles, mapBr for the 32 narrower ones).
template <int EPI, bool WIDE = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tp_gemm_pair_kernel(const __grid_constant__ CUtensorMap mapA,
                        const __grid_constant__ CUtensorMap mapB,
                        const __grid_constant__ CUtensorMap mapO,
                        const __grid_constant__ CUtensorMap mapB2,
                        const __grid_constant__ CUtensorMap mapBr, const GemmArgs g) {
  static_assert(!WIDE || EPI == EPI_F32 || EPI == EPI_F32_RESID, "the wide schedule has the float32 epilogues only");
  constexpr int STAGES = pair_stages<EPI, WIDE>();
  constexpr int BN = kPairBN;
  constexpr uint32_t A_BYTES = 128 * BK * 2;
  constexpr uint32_t B_BYTES = pair_b_bytes<WIDE>();
  constexpr uint32_t TMEM_COLS = 512;
  constexpr uint32_t IDESC = idesc_bf16_f32(256, BN);
  constexpr int kReleaseArrivals = 8;  // 4 epilogue warps in each CTA

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + STAGES * A_BYTES;
  uint8_t *sO = sB + STAGES * B_BYTES;  // TMA-store staging: 2 buffers per epilogue warp
  uint64_t *bars = reinterpret_cast<uint64_t *>(sO + (tma_store_epi<EPI>() ? 8 * kStoreBufBytes : 0));
  // barriers: full[S] | empty[S] | tfull[kAcc] | tempty[kAcc] | drain | never
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 2 * kAcc + 2);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + kAcc + a); };
  const uint32_t drain = bar0 + 8u * (2 * STAGES + 2 * kAcc);
  const uint32_t never = drain + 8u;  // nothing ever arrives here (timeout test)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < kAcc; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), kReleaseArrivals);
    }
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&mapA);
    prefetch_tmap(&mapB);
    if constexpr (tma_store_epi<EPI>()) prefetch_tmap(&mapO);
    if constexpr (WIDE) {
      prefetch_tmap(&mapB2);
      prefetch_tmap(&mapBr);
    }
  }
  if (warp == 1) {
    tmem_alloc2(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish2();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the set-up above overlaps the previous kernel's tail; its outputs are read only from here on
  pdl_trigger();
  pdl_wait();

  const WaitCtl w{abort_flag, g.status, g.wait_limit_ns};
  const int units = WIDE ? g.m_tiles * g.wide_q : g.slots * g.m_tiles * g.n_tiles;
  const int cluster_id = static_cast<int>(blockIdx.x >> 1);
  const int nclusters = static_cast<int>(gridDim.x >> 1);

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer (both CTAs, own half of each tile) ----
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      const bool leader = rank == 0;
      constexpr bool amn = EPI == EPI_F32_MN, bmn = EPI == EPI_F32_MN;
      auto advance = [&]() {
        issued |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      };
      if constexpr (WIDE) {
        // Each unit (tile) over the whole K range: A, and B in two pieces (the second at 128
        // rows into the stage's B space).
        for (int u = cluster_id; u < units && ok; u += nclusters) {
          const WideUnit wu = decode_wide(u, g);
          const int h2 = (wu.width - 256) / 2;  // this CTA's rows of the second B piece
          const CUtensorMap *mb2 = wu.width == g.wide_bn ? &mapB2 : &mapBr;
          const int brow1 = wu.n0 + 128 * static_cast<int>(rank);
          const int brow2 = wu.n0 + 256 + h2 * static_cast<int>(rank);
          const int arow = wu.m0 * 256 + 128 * static_cast<int>(rank);
          const uint32_t tx = 2u * (A_BYTES + static_cast<uint32_t>(128 + h2) * BK * 2);  // both CTAs' bytes
          KCursor kc;
          kc.start(0, g);
          for (int kt = 0; kt < g.kt_total; ++kt, kc.next()) {
            if (!wait_bar_spin(empty_bar(stage), phase ^ 1u, w)) {
              ok = false;
              break;
            }
            int ak, az, bk, bz;
            kc.coords(g.a_seg, ak, az);
            kc.coords(g.b_seg, bk, bz);
            const uint32_t da = smem_u32(sA + stage * A_BYTES), db = smem_u32(sB + stage * B_BYTES);
            if (leader) {
              const uint32_t fb = full_bar(stage);
              mbar_arrive_expect_tx(fb, tx);
              tma_load_3d(da, &mapA, fb, ak, arow, az);
              tma_load_3d(db, &mapB, fb, bk, brow1, bz);
              tma_load_3d(db + 128 * BK * 2, mb2, fb, bk, brow2, bz);
            } else {
              const uint32_t fb = map_to_rank(full_bar(stage), 0);
              tma_load_3d_pair(da, &mapA, fb, ak, arow, az);
              tma_load_3d_pair(db, &mapB, fb, bk, brow1, bz);
              tma_load_3d_pair(db + 128 * BK * 2, mb2, fb, bk, brow2, bz);
            }
            advance();
          }
        }
      }
      for (int u = cluster_id; !WIDE && u < units && ok; u += nclusters) {
        const Unit t = decode_unit(u, g);
        const int arow = t.m * 256 + 128 * static_cast<int>(rank);
        const int brow = t.n * BN + (BN / 2) * static_cast<int>(rank);
        MnBlocks<2> ablk, bblk;  // 128 rows of A and of B in each CTA
        if constexpr (amn) ablk.set(arow, g.a_mn_seg);
        if constexpr (bmn) bblk.set(brow, g.b_mn_seg);
        KCursor kc;
        kc.start(t.kt0, g);
        for (int kt = t.kt0; kt < t.kt1; ++kt, kc.next()) {
          if (!wait_bar_spin(empty_bar(stage), phase ^ 1u, w)) {
            ok = false;
            break;
          }
          int ak, az, bk, bz;
          kc.coords(g.a_seg, ak, az);
          kc.coords(g.b_seg, bk, bz);
          if constexpr (amn) {
            // this CTA's copies complete on CTA 0's stage barrier, which CTA 0 arms for both
            const uint32_t fb = leader ? full_bar(stage) : map_to_rank(full_bar(stage), 0);
            if (leader) mbar_arrive_expect_tx(fb, 2u * (A_BYTES + B_BYTES));
            // both 64-row MN blocks of this CTA's 128 rows in one copy per operand (kMnPairBox)
            if (leader) {
              tma_load_4d(smem_u32(sA + stage * A_BYTES), &mapA, fb, 0, kc.kflat, ablk.x[0] / 64, ablk.z[0]);
              tma_load_4d(smem_u32(sB + stage * B_BYTES), &mapB, fb, 0, kc.kflat, bblk.x[0] / 64, bblk.z[0]);
            } else {
              tma_load_4d_pair(smem_u32(sA + stage * A_BYTES), &mapA, fb, 0, kc.kflat, ablk.x[0] / 64, ablk.z[0]);
              tma_load_4d_pair(smem_u32(sB + stage * B_BYTES), &mapB, fb, 0, kc.kflat, bblk.x[0] / 64, bblk.z[0]);
            }
          } else if (leader) {
            const uint32_t fb = full_bar(stage);
            mbar_arrive_expect_tx(fb, 2u * (A_BYTES + B_BYTES));
            tma_load_3d(smem_u32(sA + stage * A_BYTES), &mapA, fb, ak, arow, az);
            tma_load_3d(smem_u32(sB + stage * B_BYTES), &mapB, fb, bk, brow, bz);
          } else {
            const uint32_t fb = map_to_rank(full_bar(stage), 0);
            tma_load_3d_pair(smem_u32(sA + stage * A_BYTES), &mapA, fb, ak, arow, az);
            tma_load_3d_pair(smem_u32(sB + stage * B_BYTES), &mapB, fb, bk, brow, bz);
          }
          advance();
        }
      }
      if (!ok && issued) {
        if (leader) {
          for (int s = 0; s < STAGES; ++s)
            if ((issued >> s) & 1u) drain_bar(full_bar(s), (last_par >> s) & 1u, g.status);
        } else {
          const unsigned long long t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < kPeerDrainNs) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---- MMA issuer (CTA 0 only) ----
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = !(g.wait_limit_ns < kShortLimitNs) || wait_bar(never, 0u, w);
      constexpr bool amn = EPI == EPI_F32_MN, bmn = EPI == EPI_F32_MN;
      constexpr uint32_t idesc = IDESC | (amn ? kIdescMnA : 0u) | (bmn ? kIdescMnB : 0u);
      constexpr uint32_t astep = amn ? 128u : 2u, bstep = bmn ? 128u : 2u;
      if constexpr (WIDE) {
        // A tile's first 256 columns accumulate at TMEM column 0, the rest at 256: each k-step's
        // two MMAs write different accumulators, so neither waits for the other's result.  One
        // accumulator of up to kWideMaxN columns: a unit after the first waits until the
        // epilogue has drained the one before.
        constexpr uint32_t id1 = idesc_bf16_f32(256, 256);
        const uint32_t d = tmem_base;
        uint32_t tphase = 0;
        for (int u = cluster_id; u < units && ok; u += nclusters) {
          const WideUnit wu = decode_wide(u, g);
          const uint32_t id2 = idesc_bf16_f32(256, wu.width - 256);
          if (!wait_bar_spin(tempty_bar(0), tphase ^ 1u, w)) break;
          tc_fence_after();
          for (int kt = 0; kt < g.kt_total; ++kt) {
            if (!wait_bar_spin(full_bar(stage), phase, w)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(sA + stage * A_BYTES), sb = smem_u32(sB + stage * B_BYTES);
            const uint64_t ad = sw128_kmajor_desc(sa), bd = sw128_kmajor_desc(sb);
            const uint64_t bd2 = sw128_kmajor_desc(sb + 128 * BK * 2);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint32_t accum = (kt > 0 || k > 0) ? 1u : 0u;
              tc_mma2_bf16(d, ad + 2u * k, bd + 2u * k, id1, accum);
              tc_mma2_bf16(d + 256u, ad + 2u * k, bd2 + 2u * k, id2, accum);
            }
            tc_commit2_multicast(empty_bar(stage), 0x3);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit2_multicast(tfull_bar(0), 0x3);
          tphase ^= 1u;
        }
      }
      for (int u = cluster_id; !WIDE && u < units && ok; u += nclusters) {
        const Unit t = decode_unit(u, g);
        if (!wait_bar_spin(tempty_bar(acc), acc_phase ^ 1u, w)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kt = t.kt0; kt < t.kt1; ++kt) {
          if (!wait_bar_spin(full_bar(stage), phase, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(sA + stage * A_BYTES), sb = smem_u32(sB + stage * B_BYTES);
          const uint64_t ad = amn ? sw128_mnmajor_desc(sa) : sw128_kmajor_desc(sa);
          const uint64_t bd = bmn ? sw128_mnmajor_desc(sb) : sw128_kmajor_desc(sb);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma2_bf16(d, ad + astep * k, bd + bstep * k, idesc, (kt > t.kt0 || k > 0) ? 1u : 0u);
          tc_commit2_multicast(empty_bar(stage), 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit2_multicast(tfull_bar(acc), 0x3);
        if (++acc == kAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      tc_commit2(drain);
      drain_bar(drain, 0u, g.status);
    }
    __syncwarp();
  } else {
    // ---- epilogue (warps 2..5 of both CTAs) ----
    const int q = warp & 3;
    const int row_in_tile = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t nstore = 0;  // TMA-store chunks this warp issued
    if constexpr (WIDE) {
      uint32_t tphase = 0;
      for (int u = cluster_id; u < units; u += nclusters) {
        const WideUnit wu = decode_wide(u, g);
        const bool ok = wait_bar_cluster(tfull_bar(0), tphase, w);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        if constexpr (EPI == EPI_F32)
          epilogue_f32_cols(tb, wu.n0, wu.width, wu.m0 * 256 + 128 * static_cast<int>(rank) + q * 32, lane, g,
                            &mapO, sO + q * 2 * kStoreBufBytes, nstore);
        else
          epilogue_resid_cols(tb, wu.m0 * 256 + 128 * static_cast<int>(rank) + row_in_tile, wu.n0, wu.width, g);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(map_to_rank(tempty_bar(0), 0));
        tphase ^= 1u;
      }
    }
    for (int u = cluster_id; !WIDE && u < units; u += nclusters) {
      const Unit t = decode_unit(u, g);
      const bool ok = wait_bar_cluster(tfull_bar(acc), acc_phase, w);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(acc * BN);
      if constexpr (tma_store_epi<EPI>())
        epilogue_tile_tma<BN, EPI>(tb, t, t.m * 256 + 128 * static_cast<int>(rank) + q * 32, lane, g, &mapO,
                                   sO + q * 2 * kStoreBufBytes, nstore);
      else
        epilogue_tile<BN, EPI>(tb, t, t.m * 256 + 128 * static_cast<int>(rank), row_in_tile, g);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_rank(tempty_bar(acc), 0));
      if (++acc == kAcc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // the staging buffers must outlive the stores that read them
    if (tma_store_epi<EPI>() && lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc2(tmem_base, TMEM_COLS);
  }
}

// Launch as a programmatic dependent of the previous kernel on the stream: the kernel's
// set-up (barriers, TMEM, tensor-map prefetch) runs while that kernel finishes, and
// pdl_wait in the kernel orders everything after it behind that kernel's completion.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), dim3 grid, size_t smem, cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Clusters of the pair kernel <EPI, WIDE> that fit on the GPU at once (pairs of SMs with room for
// one CTA each), per device, found on the first launch there (one array per instantiation).
// Atomic, as host threads may launch concurrently; they would store the same value.
template <int EPI, bool WIDE>
int pair_capacity(int num_sms) {
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::atomic<int> &slot = max_clusters[dev & 63];
  int mc = slot.load(std::memory_order_relaxed);
  if (mc <= 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = pair_smem_bytes<EPI, WIDE>();
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tp_gemm_pair_kernel<EPI, WIDE>, &cfg) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      n = num_sms / 2;
    }
    mc = n;
    slot.store(n, std::memory_order_relaxed);
  }
  return mc;
}

template <int EPI, bool WIDE = false>
cudaError_t launch_pair(const CUtensorMap &a, const CUtensorMap &b, const GemmArgs &g, int num_sms,
                        cudaStream_t stream, const CUtensorMap *b2 = nullptr, const CUtensorMap *br = nullptr) {
  constexpr size_t smem = pair_smem_bytes<EPI, WIDE>();
  auto kern = tp_gemm_pair_kernel<EPI, WIDE>;
  CUtensorMap o;
  std::memset(&o, 0, sizeof o);
  if constexpr (tma_store_epi<EPI>()) {
    // the output as [segments][rows][columns]: float32 slots, or the bf16 per-shard Y buffers
    bool ok;
    const uint64_t rows = static_cast<uint64_t>(g.rows_valid);
    if constexpr (EPI == EPI_F32) {
      const uint64_t ld = static_cast<uint64_t>(g.ld_out) * 4;
      const uint64_t ss = g.slots > 1 ? static_cast<uint64_t>(g.slot_stride) * 4 : rows * ld;
      ok = encode_store_map(&o, g.out, 4, static_cast<uint64_t>(g.ld_out), rows, static_cast<uint64_t>(g.slots), ld,
                            ss, 32, 32);
    } else {
      const uint64_t shards = static_cast<uint64_t>(g.cols_valid / g.shard_cols);
      ok = encode_store_map(&o, g.out, 2, static_cast<uint64_t>(g.shard_cols), rows, shards,
                            static_cast<uint64_t>(g.ld_out) * 2, static_cast<uint64_t>(g.shard_stride) * 2, 64, 32);
    }
    if (!ok) return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long units = WIDE ? static_cast<long long>(g.m_tiles) * g.wide_q
                               : static_cast<long long>(g.slots) * g.m_tiles * g.n_tiles;
  if (units <= 0) return cudaSuccess;
  const int mc = pair_capacity<EPI, WIDE>(num_sms);
  const int clusters = static_cast<int>(units < mc ? units : mc);
  return launch_dependent(kern, dim3(2 * clusters), smem, stream, a, b, o, b2 ? *b2 : b, br ? *br : b, g);
}

template <int BN, int EPI>
cudaError_t launch_impl(const CUtensorMap &a, const CUtensorMap &b, const GemmArgs &g, int num_sms,
                        cudaStream_t stream) {
  constexpr size_t smem = smem_bytes<BN>();
  auto kern = tp_gemm_kernel<BN, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long units = static_cast<long long>(g.slots) * g.m_tiles * g.n_tiles;
  if (units <= 0) return cudaSuccess;
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  return launch_dependent(kern, dim3(grid), smem, stream, a, b, g);
}

}  // namespace
}  // namespace gemm_impl
}  // namespace tp
