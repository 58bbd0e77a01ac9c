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
// are visited 128 at a time and the scores never leave the SM:
//   warp 0      TMA producer: the Q tile once per unit; K and V^T tiles of
//               128 keys through two 2-deep rings, keys one tile ahead of
//               values (S needs only K, P V only V);
//   warp 1      TMEM allocation; one thread issues S_j = Q K_j^T (128 x 128,
//               K = 128) into a double-buffered TMEM tile and, once the
//               softmax threads have written P_j, O += P_j V_j (128 x 128,
//               K = 128 keys) into the output accumulator, also in TMEM;
//   warps 2..5  one thread per query row (TMEM lane = row): the row of S_j
//               into registers, its maximum, P_j = 2^(t - m_r) as bf16 into
//               a double-buffered shared tile in the 128-byte-swizzled
//               K-major layout the MMA reads, and the row sum.
// The shift m_r is raised only when a tile's maximum exceeds it by more than
// 8 (so P <= 2^8): then the row's sum and its accumulator are scaled by
// 2^(m_old - m_new) once the previous P V has completed.  After the first
// tiles this is rare, so the accumulator normally stays with the tensor core.
// Units run heaviest first (causal: the last query tiles) and are dealt to
// the CTAs in snake order, so CTA loads stay even.  Every wait is bounded
// like the GEMM's; on a timeout the CTA drains what it issued and reports
// through the status word.
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
constexpr int kBars = 24;
constexpr float kRescaleGap = 8.0f;       // log2 of the largest unnormalised probability

// Q | K[2] | Vt[2] | P[2] | barriers
constexpr size_t kSmemBytes = 1024 + 7 * static_cast<size_t>(kTileBytes) + kBars * 8 + 16;
static_assert(kSmemBytes <= 232448, "attention tiles exceed the shared memory of one CTA");

// TMEM columns: S[0] 0..127, S[1] 128..255, O 256..383
constexpr uint32_t kOcol = 256;

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

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                    const __grid_constant__ CUtensorMap mapVt, const AttnArgs a) {
  constexpr uint32_t IDESC = idesc_bf16_f32(128, 128);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem;
  uint8_t *sK = sQ + kTileBytes;      // 2 tiles
  uint8_t *sV = sK + 2 * kTileBytes;  // 2 tiles
  uint8_t *sP = sV + 2 * kTileBytes;  // 2 tiles
  uint64_t *bars = reinterpret_cast<uint64_t *>(sP + 2 * kTileBytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kBars);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
  const uint32_t b0 = smem_u32(bars);
  // barrier i at b0 + 8 i
  const uint32_t q_full = b0, q_empty = b0 + 8;
  auto k_full = [&](int s) { return b0 + 16 + 8u * s; };
  auto k_empty = [&](int s) { return b0 + 32 + 8u * s; };
  auto v_full = [&](int s) { return b0 + 48 + 8u * s; };
  auto v_empty = [&](int s) { return b0 + 64 + 8u * s; };
  auto s_full = [&](int s) { return b0 + 80 + 8u * s; };
  auto s_empty = [&](int s) { return b0 + 96 + 8u * s; };
  auto p_full = [&](int s) { return b0 + 112 + 8u * s; };
  auto p_empty = [&](int s) { return b0 + 128 + 8u * s; };
  const uint32_t pv_done = b0 + 144;  // one phase per P V product, in issue order
  const uint32_t o_free = b0 + 152;   // one phase per unit: the accumulator has been read out
  const uint32_t drain = b0 + 160, never = b0 + 168;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
      mbar_init(s_full(s), 1);
      mbar_init(s_empty(s), kSoftmaxThreads);
      mbar_init(p_full(s), kSoftmaxThreads);
      mbar_init(p_empty(s), 1);
    }
    mbar_init(pv_done, 1);
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
      bool ok = true;
      auto load_k = [&](const AttnUnit &t, int j) -> bool {
        const int st = kc & 1;
        if (!wait_bar(k_empty(st), ((kc >> 1) & 1u) ^ 1u, w)) return false;
        mbar_arrive_expect_tx(k_full(st), kTileBytes);
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d(smem_u32(sK + st * kTileBytes + kb * kSub), &mapK, k_full(st), kb * 64, j * kTile, t.head);
        ++kc;
        return true;
      };
      auto load_v = [&](const AttnUnit &t, int j) -> bool {
        const int st = vc & 1;
        if (!wait_bar(v_empty(st), ((vc >> 1) & 1u) ^ 1u, w)) return false;
        mbar_arrive_expect_tx(v_full(st), kTileBytes);
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d(smem_u32(sV + st * kTileBytes + kb * kSub), &mapVt, v_full(st), j * kTile + kb * 64, 0,
                      t.head);
        ++vc;
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int u = unit_of(k, b, G);
        if (u >= units) break;
        const AttnUnit t = decode(u, a);
        if (!wait_bar(q_empty, (qc & 1u) ^ 1u, w)) break;
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
      for (int s = 0; s < 2; ++s) {
        const int nk = (kc - s + 1) / 2, nv = (vc - s + 1) / 2;  // loads issued into stage s
        if (nk > 0) drain_bar(k_full(s), (nk - 1) & 1u, a.status);
        if (nv > 0) drain_bar(v_full(s), (nv - 1) & 1u, a.status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer ----
      int sc = 0, pc = 0, uc = 0;  // S tiles issued, P V products issued, units started
      bool ok = !(a.wait_limit_ns < kShortLimitNs) || wait_bar(never, 0u, w);
      auto issue_s = [&]() -> bool {
        // S[sc & 1] = Q K^T over head_dim 128: two 64-wide sub-tiles x four K = 16 steps
        const int st = sc & 1;
        const uint32_t ph = (sc >> 1) & 1u;
        if (!wait_bar(k_full(st), ph, w) || !wait_bar(s_empty(st), ph ^ 1u, w)) return false;
        tc_fence_after();
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          const uint64_t ad = sw128_kmajor_desc(smem_u32(sQ + kb * kSub));
          const uint64_t bd = sw128_kmajor_desc(smem_u32(sK + st * kTileBytes + kb * kSub));
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc_mma_bf16(tmem + st * 128, ad + 2u * k, bd + 2u * k, IDESC, (kb | k) ? 1u : 0u);
        }
        tc_commit(s_full(st));
        tc_commit(k_empty(st));
        ++sc;
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int u = unit_of(k, b, G);
        if (u >= units) break;
        const AttnUnit t = decode(u, a);
        if (!wait_bar(q_full, uc & 1u, w)) break;
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
          // O += P_j V_j once the softmax threads have written P_j (and, for the
          // first key tile, read out the previous unit's O)
          const int st = pc & 1;
          const uint32_t ph = (pc >> 1) & 1u;
          if (!wait_bar(p_full(st), ph, w) || !wait_bar(v_full(st), ph, w) ||
              (j == 0 && !wait_bar(o_free, (uc & 1u) ^ 1u, w))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
            const uint64_t ad = sw128_kmajor_desc(smem_u32(sP + st * kTileBytes + kb * kSub));
            const uint64_t bd = sw128_kmajor_desc(smem_u32(sV + st * kTileBytes + kb * kSub));
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc_mma_bf16(tmem + kOcol, ad + 2u * k, bd + 2u * k, IDESC, (j | kb | k) ? 1u : 0u);
          }
          tc_commit(pv_done);
          tc_commit(p_empty(st));
          tc_commit(v_empty(st));
          ++pc;
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
    const int sw = row_in_tile & 7;  // 128-byte swizzle: 16-byte chunk q of this row sits at q ^ sw
    int kt = 0;  // key tiles consumed by this CTA (S and P buffers and P V products count with it)
    bool ok = true;
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool got = wait_bar(bar, parity, w);
      return __all_sync(0xffffffffu, got);
    };
    for (int k = 0; ok; ++k) {
      const int u = unit_of(k, b, G);
      if (u >= units) break;
      const AttnUnit t = decode(u, a);
      const int row = t.mt * kTile + row_in_tile;
      float m_used = -INFINITY, l_run = 0.f;
      for (int j = 0; j < t.nkt; ++j) {
        const int idx = kt + j;
        const int st = idx & 1;
        const uint32_t ph = (idx >> 1) & 1u;
        if (!wait_all(s_full(st), ph)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the row of S_j: 128 scores in registers, then the S buffer is free
        uint32_t s[4][32];
        const uint32_t sb = tmem + lane_base + st * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(sb + cc * 32, s[cc]);
        tmem_ld_wait();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_reg_fence(s[cc]);
        tc_fence_before();
        mbar_arrive(s_empty(st));
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
        for (int q = 0; q < 8; ++q) mx8[q] = __uint_as_float(s[q >> 1][(q & 1) * 16]);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int q = cc * 2 + i / 16;
            if (i % 16 != 0) mx8[q] = fmaxf(mx8[q], __uint_as_float(s[cc][i]));
          }
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        const float m_tile = mx * c;
        const bool raise = m_tile > m_used + kRescaleGap;
        const float m_new = raise ? m_tile : m_used;
        const float alpha = raise ? ex2_approx(m_used - m_new) : 1.0f;  // 0 on the first tile
        m_used = m_new;
        // P = 2^(t - m) as bf16 into P[st] (free once the P V of key tile idx - 2 is done)
        if (!wait_all(p_empty(st), ph ^ 1u)) {
          ok = false;
          break;
        }
        uint8_t *prow = sP + st * kTileBytes + row_in_tile * 128;
        float sum8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) sum8[q] = 0.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            // keys 32 cc + 8 h .. + 7: one 16-byte chunk (chunk 4 (cc & 1) + h of sub-tile cc / 2)
            // the row sum adds the bf16-rounded weights the P V product uses, so each
            // output is a convex combination of the values (rounding of P cancels)
            uint32_t pk[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              pk[i] = pack_bf16x2(ex2_approx(fmaf(__uint_as_float(s[cc][8 * h + 2 * i]), c, -m_new)),
                                  ex2_approx(fmaf(__uint_as_float(s[cc][8 * h + 2 * i + 1]), c, -m_new)));
              sum8[2 * i] += __uint_as_float(pk[i] << 16);
              sum8[2 * i + 1] += __uint_as_float(pk[i] & 0xFFFF0000u);
            }
            const int chunk = (cc & 1) * 4 + h;
            *reinterpret_cast<uint4 *>(prow + (cc >> 1) * kSub + ((chunk ^ sw) << 4)) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
        const float sum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
        l_run = fmaf(l_run, alpha, sum);
        // a raised shift also scales the accumulated O, once the previous P V is in it
        // (P V of key tile idx - 2 is done: P[st] was released above)
        if (j > 0 && __any_sync(0xffffffffu, raise)) {
          if (!wait_all(pv_done, (idx - 1) & 1u)) {
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
          tmem_st_wait();
        }
        tc_fence_before();
        fence_proxy_async_smem();
        mbar_arrive(p_full(st));
      }
      if (!ok) break;
      // read out O / l once the unit's last P V is done.  A parity wait names the
      // current or the preceding phase only, so wait for the last two products in
      // turn (the one before them is known to be done: its P buffer was released).
      const int last = kt + t.nkt - 1;
      if ((t.nkt > 1 && !wait_all(pv_done, (last - 1) & 1u)) || !wait_all(pv_done, last & 1u)) break;
      tc_fence_after();
      kt += t.nkt;
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
