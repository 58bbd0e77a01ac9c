// tp_attention.cu - fused attention core of the tensor-parallel transformer
// block ("Tensor parallelism" guide, section "Walking through a transformer
// block": heads are sharded across ranks, so each head's attention is local
// to the shard that owns it and needs no communication).
//
// One CTA per SM walks units (head, 128-query tile) and computes, for each
// query row r of the tile,
//   O[r] = sum_{j allowed} 2^(t_rj - m_r) v_j / sum_{j allowed} 2^(t_rj - m_r),
//   t_rj = (q_r . k_j / sqrt(128)) log2(e),
// which is the softmax-weighted sum of the values for any shift m_r.  Keys
// are visited 128 at a time and neither scores nor probabilities leave the
// SM, or even reach shared memory:
//   warp 0      TMA producer: the Q tile once per unit; K and V^T tiles of
//               128 keys through two 3-deep rings, keys one tile ahead of
//               values (S needs only K, P V only V);
//   warp 1      TMEM allocation; one thread issues S_j = Q K_j^T (128 x 128,
//               K = 128, both operands in shared memory) into one of three
//               TMEM buffers and, once the softmax threads have overwritten
//               that buffer's first 64 columns with P_j (bf16 pairs),
//               O += P_j V_j with P_j read from TMEM (128 x 128, K = 128 keys)
//               into the output accumulator, also in TMEM;
//   warps 2..5  one thread per query row (TMEM lane = row): the row of S_j
//               into registers, its maximum, P_j = 2^(t - m_r) rounded to
//               bf16 back into TMEM, and the row sum of those rounded weights.
// The shift m_r is raised only when a tile's maximum exceeds it by more than
// 8 (so P <= 2^8): then the row's sum and its accumulator are scaled by
// 2^(m_old - m_new) once the previous P V has completed.  After the first
// tiles this is rare, so the accumulator normally stays with the tensor core.
// Units run heaviest first (causal: the last query tiles) and are dealt to
// the CTAs in snake order, so CTA loads stay even.  Waits poll (the S ->
// softmax -> P V round trip is on the critical path, and a suspended wait
// wakes too late) and are bounded like the GEMM's; on a timeout the CTA
// drains what it issued and reports through the status word.
#include <cuda_bf16.h>

#include "tp_device.cuh"
#include "tp_internal.h"

namespace tp {
namespace {

constexpr int kTile = 128;                // queries per unit, keys per step
constexpr int kThreads = 192;
constexpr int kSoftmaxThreads = 128;
constexpr uint32_t kSub = 128 * 128;      // 128 rows x 64 bf16, swizzled (16 KiB)
constexpr uint32_t kTileBytes = 2 * kSub; // 128 x 128 bf16
constexpr int kSbuf = 3;                  // S / P buffers in TMEM
constexpr int kKst = 3, kVst = 3;         // K and V^T tiles in shared memory
constexpr int kBars = 28;
constexpr float kRescaleGap = 8.0f;       // log2 of the largest unnormalised probability

// Q | K[kKst] | Vt[kVst] | barriers
constexpr size_t kSmemBytes = 1024 + (1 + kKst + kVst) * static_cast<size_t>(kTileBytes) + kBars * 8 + 16;
static_assert(kSmemBytes <= 232448, "attention tiles exceed the shared memory of one CTA");

// TMEM columns: S/P buffers 0..383 (128 each), O 384..511
constexpr uint32_t kOcol = kSbuf * 128;

struct AttnUnit {
  int head, mt, nkt;  // head, query tile, key tiles to visit
};

// k-th unit of CTA b among G CTAs: snake order over the heaviest-first list.
__device__ __forceinline__ int unit_of(int k, int b, int G) { return k * G + ((k & 1) ? G - 1 - b : b); }

__device__ __forceinline__ AttnUnit decode(int u, const AttnArgs &a) {
  AttnUnit t;
  t.mt = a.m_tiles - 1 - u / a.heads;
  t.head = u % a.heads;
  t.nkt = a.causal ? t.mt + 1 : a.m_tiles;
  return t;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Position in a ring of n buffers: buffer index and phase parity, stepped per use.
struct Ring {
  int buf = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++buf == n) {
      buf = 0;
      phase ^= 1u;
    }
  }
};

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                    const __grid_constant__ CUtensorMap mapVt, const AttnArgs a) {
  constexpr uint32_t IDESC = idesc_bf16_f32(128, 128);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem;
  uint8_t *sK = sQ + kTileBytes;
  uint8_t *sV = sK + kKst * kTileBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sV + kVst * kTileBytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kBars);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
  const uint32_t b0 = smem_u32(bars);
  // barrier i at b0 + 8 i
  const uint32_t q_full = b0, q_empty = b0 + 8;
  auto k_full = [&](int s) { return b0 + 16 + 8u * s; };    // kKst
  auto k_empty = [&](int s) { return b0 + 40 + 8u * s; };   // kKst
  auto v_full = [&](int s) { return b0 + 64 + 8u * s; };    // kVst
  auto v_empty = [&](int s) { return b0 + 88 + 8u * s; };   // kVst
  auto s_full = [&](int s) { return b0 + 112 + 8u * s; };   // S_j computed (kSbuf)
  // the P V that read P from it is done; as each commit covers every earlier MMA, also
  // "all P V products up to that one are in O" (kSbuf)
  auto s_empty = [&](int s) { return b0 + 136 + 8u * s; };
  auto p_full = [&](int s) { return b0 + 160 + 8u * s; };   // P_j written over S_j (kSbuf)
  const uint32_t o_free = b0 + 184;   // one phase per unit: the accumulator has been read out
  const uint32_t drain = b0 + 192, never = b0 + 200;
  static_assert(kKst <= 3 && kVst <= 3 && kSbuf <= 3 && 26 <= kBars, "barrier layout");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kKst; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < kVst; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int s = 0; s < kSbuf; ++s) {
      mbar_init(s_full(s), 1);
      mbar_init(s_empty(s), 1);
      mbar_init(p_full(s), kSoftmaxThreads);
    }
    mbar_init(o_free, kSoftmaxThreads);
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&mapQ);
    prefetch_tmap(&mapK);
    prefetch_tmap(&mapVt);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl w{abort_flag, a.status, a.wait_limit_ns};
  const int units = a.heads * a.m_tiles;
  const int G = gridDim.x, b = blockIdx.x;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer ----
      // Loads per unit, in order: Q, K_0, then for each j: K_{j+1} (if any), V_j.
      int kc = 0, vc = 0, qc = 0;  // K, V tiles and Q tiles issued so far
      Ring kr, vr;
      bool ok = true;
      auto load_k = [&](const AttnUnit &t, int j) -> bool {
        if (!wait_bar_spin(k_empty(kr.buf), kr.phase ^ 1u, w)) return false;
        mbar_arrive_expect_tx(k_full(kr.buf), kTileBytes);
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d(smem_u32(sK + kr.buf * kTileBytes + kb * kSub), &mapK, k_full(kr.buf), kb * 64, j * kTile,
                      t.head);
        ++kc;
        kr.next(kKst);
        return true;
      };
      auto load_v = [&](const AttnUnit &t, int j) -> bool {
        if (!wait_bar_spin(v_empty(vr.buf), vr.phase ^ 1u, w)) return false;
        mbar_arrive_expect_tx(v_full(vr.buf), kTileBytes);
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d(smem_u32(sV + vr.buf * kTileBytes + kb * kSub), &mapVt, v_full(vr.buf), j * kTile + kb * 64,
                      0, t.head);
        ++vc;
        vr.next(kVst);
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int u = unit_of(k, b, G);
        if (u >= units) break;
        const AttnUnit t = decode(u, a);
        if (!wait_bar_spin(q_empty, (qc & 1u) ^ 1u, w)) break;
        mbar_arrive_expect_tx(q_full, kTileBytes);
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d(smem_u32(sQ + kb * kSub), &mapQ, q_full, kb * 64, t.mt * kTile, t.head);
        ++qc;
        if (!load_k(t, 0)) break;
        for (int j = 0; j < t.nkt; ++j) {
          if (j + 1 < t.nkt && !load_k(t, j + 1)) {
            ok = false;
            break;
          }
          if (!load_v(t, j)) {
            ok = false;
            break;
          }
        }
      }
      // Every copy issued completes on its full barrier, consumed or not (after an abort
      // some are not): wait for the last phase of each before the CTA may exit.
      if (qc > 0) drain_bar(q_full, (qc - 1) & 1u, a.status);
      for (int s = 0; s < kKst; ++s) {
        const int n = (kc - s + kKst - 1) / kKst;  // loads issued into stage s
        if (n > 0) drain_bar(k_full(s), (n - 1) & 1u, a.status);
      }
      for (int s = 0; s < kVst; ++s) {
        const int n = (vc - s + kVst - 1) / kVst;
        if (n > 0) drain_bar(v_full(s), (n - 1) & 1u, a.status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer ----
      int uc = 0;           // units started
      Ring kr, vr, sr, pr;  // K tile and S buffer of the next S; V tile and S buffer of the next P V
      bool ok = !(a.wait_limit_ns < kShortLimitNs) || wait_bar_spin(never, 0u, w);
      auto issue_s = [&]() -> bool {
        // S = Q K^T over head_dim 128: two 64-wide sub-tiles x four K = 16 steps
        if (!wait_bar_spin(k_full(kr.buf), kr.phase, w) || !wait_bar_spin(s_empty(sr.buf), sr.phase ^ 1u, w))
          return false;
        tc_fence_after();
        const uint32_t d = tmem + sr.buf * 128;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          const uint64_t ad = sw128_kmajor_desc(smem_u32(sQ + kb * kSub));
          const uint64_t bd = sw128_kmajor_desc(smem_u32(sK + kr.buf * kTileBytes + kb * kSub));
#pragma unroll
          for (int k = 0; k < 4; ++k) tc_mma_bf16(d, ad + 2u * k, bd + 2u * k, IDESC, (kb | k) ? 1u : 0u);
        }
        tc_commit(s_full(sr.buf));
        tc_commit(k_empty(kr.buf));
        kr.next(kKst);
        sr.next(kSbuf);
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int u = unit_of(k, b, G);
        if (u >= units) break;
        const AttnUnit t = decode(u, a);
        if (!wait_bar_spin(q_full, uc & 1u, w)) break;
        tc_fence_after();
        if (!issue_s()) break;
        for (int j = 0; j < t.nkt; ++j) {
          if (j + 1 < t.nkt) {
            if (!issue_s()) {
              ok = false;
              break;
            }
          } else {
            tc_commit(q_empty);  // every S of this unit is issued: Q may be replaced
          }
          // O += P_j V_j once the softmax threads have written P_j over S_j (and, for the
          // first key tile, read out the previous unit's O)
          if (!wait_bar_spin(p_full(pr.buf), pr.phase, w) || !wait_bar_spin(v_full(vr.buf), vr.phase, w) ||
              (j == 0 && !wait_bar_spin(o_free, (uc & 1u) ^ 1u, w))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t pa = tmem + pr.buf * 128;  // P: 64 columns of bf16 pairs
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t bd = sw128_kmajor_desc(smem_u32(sV + vr.buf * kTileBytes + (kk >> 2) * kSub));
            tc_mma_bf16_tmem_a(tmem + kOcol, pa + 8u * kk, bd + 2u * (kk & 3), IDESC, (j | kk) ? 1u : 0u);
          }
          tc_commit(s_empty(pr.buf));
          tc_commit(v_empty(vr.buf));
          vr.next(kVst);
          pr.next(kSbuf);
        }
        ++uc;
      }
      tc_commit(drain);
      drain_bar(drain, 0u, a.status);
    }
    __syncwarp();
  } else {
    // ---- softmax and output (warp w reads TMEM lanes 32 (w % 4) .. + 31) ----
    const int row_in_tile = (warp & 3) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t ob = tmem + lane_base + kOcol;
    const float c = a.scale_log2;
    Ring sr, prv;  // S / P buffer of the current key tile, of the previous one
    bool ok = true;
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool got = wait_bar_spin(bar, parity, w);
      return __all_sync(0xffffffffu, got);
    };
    for (int k = 0; ok; ++k) {
      const int u = unit_of(k, b, G);
      if (u >= units) break;
      const AttnUnit t = decode(u, a);
      const int row = t.mt * kTile + row_in_tile;
      float m_used = -INFINITY, l_run = 0.f;
      for (int j = 0; j < t.nkt; prv = sr, ++j, sr.next(kSbuf)) {
        if (!wait_all(s_full(sr.buf), sr.phase)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the row of S_j: 128 scores in registers
        uint32_t s[4][32];
        const uint32_t sb = tmem + lane_base + sr.buf * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(sb + cc * 32, s[cc]);
        tmem_ld_wait();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_reg_fence(s[cc]);
        // allowed keys of this tile: key0 + i for i <= kmax (causal: key <= row; always key < M)
        const int key0 = j * kTile;
        int kmax = a.M - 1 - key0;
        if (a.causal && row - key0 < kmax) kmax = row - key0;
        if (kmax < kTile - 1) {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (cc * 32 + i > kmax) s[cc][i] = __float_as_uint(-INFINITY);
        }
        // row maximum: eight independent chains
        float mx8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float m = __uint_as_float(s[q >> 1][(q & 1) * 16]);
#pragma unroll
          for (int i = 1; i < 16; ++i) m = fmaxf(m, __uint_as_float(s[q >> 1][(q & 1) * 16 + i]));
          mx8[q] = m;
        }
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        const float m_tile = mx * c;
        const bool raise = m_tile > m_used + kRescaleGap;
        const float m_new = raise ? m_tile : m_used;
        const float alpha = raise ? ex2_approx(m_used - m_new) : 1.0f;  // 0 on the first tile
        m_used = m_new;
        // P = 2^(t - m) as bf16 pairs over the first 64 columns of the S buffer.  The row
        // sum adds the rounded weights the P V product uses, so each output is a convex
        // combination of the values (the rounding of P cancels in it).
        float sum8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) sum8[q] = 0.f;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t pk[32];  // keys 64 hh .. 64 hh + 63
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int key = 64 * hh + 2 * i;
            pk[i] = pack_bf16x2(ex2_approx(fmaf(__uint_as_float(s[key >> 5][key & 31]), c, -m_new)),
                                ex2_approx(fmaf(__uint_as_float(s[key >> 5][(key & 31) + 1]), c, -m_new)));
            sum8[(2 * i) & 7] += __uint_as_float(pk[i] << 16);
            sum8[(2 * i + 1) & 7] += __uint_as_float(pk[i] & 0xFFFF0000u);
          }
          tmem_st32(sb + hh * 32, pk);
        }
        const float sum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
        l_run = fmaf(l_run, alpha, sum);
        // a raised shift also scales the accumulated O, once the previous P V is in it.  The
        // P V before that in the same buffer is done (S_{j-1} was computed into the buffer
        // after it), so the parity wait below names the current or the preceding phase.
        if (j > 0 && __any_sync(0xffffffffu, raise)) {
          if (!wait_all(s_empty(prv.buf), prv.phase)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t r[32];
            tmem_ld32(ob + cc * 32, r);
            tmem_ld_wait();
            tmem_reg_fence(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(ob + cc * 32, r);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full(sr.buf));
      }
      if (!ok) break;
      // read out O / l once the unit's last P V (and so every earlier one) is done
      if (!wait_all(s_empty(prv.buf), prv.phase)) break;
      tc_fence_after();
      const float inv = 1.0f / l_run;
      uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.O) + static_cast<long long>(row) * a.ldo +
                                             static_cast<long long>(t.head) * kAttnHeadDim);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t r[32];
        tmem_ld32(ob + cc * 32, r);
        tmem_ld_wait();
        tmem_reg_fence(r);
        if (row < a.M) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[cc * 4 + q] = make_uint4(
                pack_bf16x2(__uint_as_float(r[8 * q]) * inv, __uint_as_float(r[8 * q + 1]) * inv),
                pack_bf16x2(__uint_as_float(r[8 * q + 2]) * inv, __uint_as_float(r[8 * q + 3]) * inv),
                pack_bf16x2(__uint_as_float(r[8 * q + 4]) * inv, __uint_as_float(r[8 * q + 5]) * inv),
                pack_bf16x2(__uint_as_float(r[8 * q + 6]) * inv, __uint_as_float(r[8 * q + 7]) * inv));
        }
      }
      tc_fence_before();
      mbar_arrive(o_free);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_attention(const CUtensorMap &mapQ, const CUtensorMap &mapK, const CUtensorMap &mapVt,
                             const AttnArgs &args, int num_sms, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const long long units = static_cast<long long>(args.heads) * args.m_tiles;
  if (units <= 0) return cudaSuccess;
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  attn_fwd_kernel<<<grid, kThreads, kSmemBytes, stream>>>(mapQ, mapK, mapVt, args);
  return cudaGetLastError();
}

}  // namespace tp
