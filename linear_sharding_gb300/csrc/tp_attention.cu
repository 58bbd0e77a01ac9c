// tp_attention.cu - fused attention core of the tensor-parallel transformer
// block ("Tensor parallelism" guide, section "Walking through a transformer
// block": heads are sharded across ranks, so each head's attention is local
// to the shard that owns it and needs no communication).
//
// One CTA per SM walks units (head, 128-query tile) and computes, for each
// query row r,
//   O[r] = sum_{j allowed} 2^(t_rj - m_r) v_j / sum_{j allowed} 2^(t_rj - m_r),
//   t_rj = (q_r . k_j / sqrt(128)) log2(e),
// which is the softmax-weighted sum of the values for any shift m_r.  Keys
// are visited 128 at a time and neither scores nor probabilities leave the
// SM, or even reach shared memory:
//   warp 4      TMA producer: the Q tile once per unit; K and V tiles of 128
//               keys through 3-deep rings, keys up to three tiles ahead of
//               values (odd units of a CTA walk their key tiles downwards);
//               L2 hints keep K and V (other query tiles of the head read
//               them again) and not Q.  Q, K and V are all head-major
//               [heads][M][128]; V is the P V product's B operand read
//               MN-major (its K, the key axis, is the outer one);
//   warp 5      TMEM allocation; one thread issues S_j = Q K_j^T (tcgen05,
//               128 x 128, K = 128) into one of three S/P buffers, up to three
//               key tiles ahead: the buffers form one ring over all of a
//               CTA's key steps, unit after unit, and S_{j+3} goes into the
//               buffer of S_j once P_j V_j has read it;
//   warp 6      one thread issues O += P_j V_j (P read from TMEM, V from
//               shared memory).  Two issuing threads: each one's waits and
//               commits overlap the other's MMAs, so the tensor core is fed
//               while either waits;
//   warps 0..3  softmax: one thread per query row (TMEM lane = row) reads the
//               row of S_j, takes its maximum, writes P = 2^(t - m_r) as bf16
//               over the upper 64 columns of the same buffer, and adds the
//               float32 weights to the row sum; at a unit's end it hands the
//               row sum to the output warps and goes on to the next unit;
//   warps 8..11 output: once a unit's last P V is done, read O out of tensor
//               memory as bf16 O / l (which frees it for the next unit's
//               first P V) and store it, while the softmax warps already work
//               on the next unit (warp 7 is idle).
// The softmax warpgroup runs with 248 registers a thread, the others with
// fewer (setmaxnreg), within the 168 a thread the CTA is launched with.
// With S computed ahead, the softmax of key tile j + 1 starts as soon as that
// of tile j ends: neither waits for the other's hand-off, and the tensor core
// has a whole S and P V (1024 cycles) per 128-key step beside it.  The shift
// m_r is raised only when a tile's maximum exceeds it by more than 8 (so
// P <= 2^8): then the row's sum and its accumulator are scaled by
// 2^(m_old - m_new), after the P V product issued before is complete (the
// barrier that frees its buffer says so).  Units run heaviest first (causal: the
// last query tiles) and are dealt to the CTAs in snake order.  The hand-offs
// are on the critical path, so waits probe with try_wait and no suspend hint
// (the thread wakes when the phase completes: faster than polling with
// test_wait, where a long hint woke too late); they are bounded like the
// GEMM's, and on a timeout the CTA drains what it issued and reports through
// the status word.
#include <cuda_bf16.h>

#include "tp_device.cuh"
#include "tp_internal.h"

namespace tp {
namespace {

constexpr int kTile = 128;                // queries per tile, keys per step
constexpr int kThreads = 384;             // softmax | producer, S issuer, P V issuer, idle | output
constexpr int kSoftmaxThreads = 128;
constexpr int kOutThreads = 128;
// registers a thread per warpgroup after setmaxnreg: softmax, issuers, output.  Their sum over
// 128 threads each (63488) stays within the launch's 384 x 168 = 64512.
constexpr int kRegsSoftmax = 248, kRegsIssue = 104, kRegsOut = 144;
static_assert(128 * (kRegsSoftmax + kRegsIssue + kRegsOut) <= kThreads * 168, "register split exceeds the launch");
constexpr int kSbuf = 3;                  // S/P buffers in tensor memory: S runs up to 3 steps ahead
constexpr uint32_t kSub = 128 * 128;      // 128 rows x 64 bf16, swizzled (16 KiB)
constexpr uint32_t kTileBytes = 2 * kSub; // 128 x 128 bf16
constexpr int kKst = 3, kVst = 3;         // K and V tiles in shared memory
static_assert(kSbuf <= kKst, "the producer copies K up to kSbuf tiles ahead, into a ring of kKst");
constexpr int kBars = 32;
constexpr float kRescaleGap = 8.0f;       // log2 of the largest unnormalised probability

// Q | K[kKst] | V[kVst] | barriers | TMEM address, abort flag | row sums (2 x 128 floats)
constexpr size_t kSmemBytes = 1024 + (1 + kKst + kVst) * static_cast<size_t>(kTileBytes) + kBars * 8 + 16 + 2 * 128 * 4;
static_assert(kSmemBytes <= 232448, "attention tiles exceed the shared memory of one CTA");

// TMEM columns: S/P buffer b at 128 b (b < 3), O at 384
constexpr uint32_t kOcol = kSbuf * 128;
static_assert(kOcol + 128 <= 512, "S/P buffers and O exceed tensor memory");

struct AttnUnit {
  int head;
  int mt;  // query tile
  int nk;  // key tiles it visits
};

// k-th unit of CTA b among G CTAs: snake order over the heaviest-first list.
__device__ __forceinline__ int unit_of(int k, int b, int G) { return k * G + ((k & 1) ? G - 1 - b : b); }

__device__ __forceinline__ AttnUnit decode(int u, const AttnArgs &a) {
  AttnUnit t;
  t.mt = a.m_tiles - 1 - u / a.heads;
  t.head = u % a.heads;
  t.nk = a.causal ? t.mt + 1 : a.m_tiles;
  if (!TP_CHECK(t.head < a.heads && t.mt >= 0 && t.nk >= 1 && t.nk <= a.m_tiles, a.status)) {
    t.mt = 0;  // keep the unit's shape sane: one key tile
    t.nk = 1;
  }
  return t;
}

// Key tile visited at key step j of a CTA's k-th unit.  Odd units walk their keys down from the
// last (causal: the diagonal) tile, so a CTA's next unit starts on the key tiles the units that
// ran just before it read last, which are still in L2: at 4096 tokens x 32 heads the DRAM reads
// fall from 152 to 111 MB (Q, K and V are 100.7 MB).  The online softmax takes the keys in any
// order.
__device__ __forceinline__ int key_tile(int k, const AttnUnit &t, int j) { return (k & 1) ? t.nk - 1 - j : j; }

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// One 32-byte global store (a whole sector); p must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t *v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]), "r"(v[1]), "r"(v[2]),
               "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
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
                    const __grid_constant__ CUtensorMap mapV, const AttnArgs a) {
  constexpr uint32_t IDESC = idesc_bf16_f32(128, 128);
  constexpr uint32_t IDESC_PV = IDESC | kIdescMnB;  // V is read MN-major: [keys][head_dim]
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem;
  uint8_t *sK = sQ + kTileBytes;
  uint8_t *sV = sK + kKst * kTileBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sV + kVst * kTileBytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kBars);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
  float *l_buf = reinterpret_cast<float *>(tmem_slot + 4);  // [2][128]: a unit's row sums
  const uint32_t b0 = smem_u32(bars);
  // barrier i at b0 + 8 i
  const uint32_t q_full = b0, q_empty = b0 + 8;
  auto k_full = [&](int s) { return b0 + 16 + 8u * s; };    // kKst
  auto k_empty = [&](int s) { return b0 + 40 + 8u * s; };   // kKst
  auto v_full = [&](int s) { return b0 + 64 + 8u * s; };    // kVst
  auto v_empty = [&](int s) { return b0 + 88 + 8u * s; };   // kVst
  auto s_full = [&](int b) { return b0 + 112 + 8u * b; };   // kSbuf: S in buffer b computed
  auto p_full = [&](int b) { return b0 + 136 + 8u * b; };   // kSbuf: P written over it
  auto s_free = [&](int b) { return b0 + 160 + 8u * b; };   // kSbuf: P V of buffer b done (P read)
  const uint32_t o_full = b0 + 184, o_free = b0 + 192;      // the unit's last P V done; O read out
  const uint32_t drain = b0 + 200, drain_pv = b0 + 208, never = b0 + 216;
  auto l_full = [&](uint32_t p) { return b0 + 224 + 8u * p; };   // 2: row sums of a unit written
  auto l_empty = [&](uint32_t p) { return b0 + 240 + 8u * p; };  // 2: row sums read

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
    for (int b = 0; b < kSbuf; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(p_full(b), kSoftmaxThreads);
      mbar_init(s_free(b), 1);
    }
    mbar_init(o_full, 1);
    mbar_init(o_free, kOutThreads);
    for (uint32_t p = 0; p < 2; ++p) {
      mbar_init(l_full(p), kSoftmaxThreads);
      mbar_init(l_empty(p), kOutThreads);
    }
    mbar_init(drain, 1);
    mbar_init(drain_pv, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tmap(&mapQ);
    prefetch_tmap(&mapK);
    prefetch_tmap(&mapV);
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the set-up above overlaps the previous kernel's tail; Q, K and V are read only from here on
  pdl_trigger();
  pdl_wait();
  const WaitCtl w{abort_flag, a.status, a.wait_limit_ns};
  const int units = a.heads * a.m_tiles;
  const int G = gridDim.x, b = blockIdx.x;
  // Roles by warpgroup; each warpgroup first takes its register share (every warp of it, at one
  // instruction; the softmax's increase waits for the others' decreases).
  if (warp >= 4 && warp < 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsIssue));
    if (warp == 4) {
      if (lane == 0) {
        // ---- TMA producer ----
        // Loads per unit, by key step: Q, the K tiles of steps 0 .. 2, then for each step j its V
        // tile and the K tile of step j + 3 (if any).
        int kc = 0, vc = 0, qc = 0;  // K, V and Q tiles issued so far
        // L2 hints: K and V tiles are read again by the other query tiles of their head (kept),
        // a Q tile by its unit only
        const uint64_t keep = policy_evict_last(), once = policy_evict_first();
        Ring kr, vr;
        bool ok = true;
        auto load_k = [&](const AttnUnit &t, int j) -> bool {
          if (!wait_bar_wake(k_empty(kr.buf), kr.phase ^ 1u, w)) return false;
          mbar_arrive_expect_tx(k_full(kr.buf), kTileBytes);
          for (int kb = 0; kb < 2; ++kb)
            tma_load_3d_hint(smem_u32(sK + kr.buf * kTileBytes + kb * kSub), &mapK, k_full(kr.buf), kb * 64, j * kTile,
                             t.head, keep);
          ++kc;
          kr.next(kKst);
          return true;
        };
        auto load_v = [&](const AttnUnit &t, int j) -> bool {
          if (!wait_bar_wake(v_empty(vr.buf), vr.phase ^ 1u, w)) return false;
          mbar_arrive_expect_tx(v_full(vr.buf), kTileBytes);
          // V_j as four 64 x 64 boxes: keys 64 h .. (16 KiB h), head_dim 64 c .. (8 KiB c)
          for (int h = 0; h < 2; ++h)
            for (int c = 0; c < 2; ++c)
              tma_load_3d_hint(smem_u32(sV + vr.buf * kTileBytes + h * kSub + c * kSub / 2), &mapV, v_full(vr.buf),
                               c * 64, j * kTile + h * 64, t.head, keep);
          ++vc;
          vr.next(kVst);
          return true;
        };
        for (int k = 0; ok; ++k) {
          const int u = unit_of(k, b, G);
          if (u >= units) break;
          const AttnUnit t = decode(u, a);
          if (!wait_bar_wake(q_empty, (qc & 1u) ^ 1u, w)) break;
          mbar_arrive_expect_tx(q_full, kTileBytes);
          for (int kb = 0; kb < 2; ++kb)
            tma_load_3d_hint(smem_u32(sQ + kb * kSub), &mapQ, q_full, kb * 64, t.mt * kTile, t.head, once);
          ++qc;
          // key step j visits key tile key_tile(k, t, j): every other unit walks down from its last
          const int pre = t.nk < kSbuf ? t.nk : kSbuf;
          for (int j = 0; j < pre && ok; ++j) ok = load_k(t, key_tile(k, t, j));
          for (int j = 0; j < t.nk && ok; ++j) {
            ok = load_v(t, key_tile(k, t, j));
            if (ok && j + kSbuf < t.nk) ok = load_k(t, key_tile(k, t, j + kSbuf));
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
    } else if (warp == 5) {
      if (lane == 0) {
        // ---- S issuer: S_j = Q K_j^T into the next buffer of the ring, once P V has read the
        // P made three key steps before in that buffer ----
        int uc = 0;                          // units started
        int sb = 0;                          // buffer of the next S (the ring runs on across units)
        Ring kr;                             // K tile of the next S
        // bit b: parity of buffer b's next s_free wait (a fresh barrier's previous phase counts as
        // complete).  Per-buffer phases live in bits of a register, not in an indexed array.
        uint32_t fph = (1u << kSbuf) - 1u;
        bool ok = !(a.wait_limit_ns < kShortLimitNs) || wait_bar_wake(never, 0u, w);
        for (int k = 0; ok; ++k) {
          const int u = unit_of(k, b, G);
          if (u >= units) break;
          const AttnUnit t = decode(u, a);
          if (!wait_bar_wake(q_full, uc & 1u, w)) break;
          for (int j = 0; j < t.nk; ++j, sb = sb + 1 == kSbuf ? 0 : sb + 1) {
            if (!wait_bar_wake(s_free(sb), (fph >> sb) & 1u, w) || !wait_bar_wake(k_full(kr.buf), kr.phase, w)) {
              ok = false;
              break;
            }
            fph ^= 1u << sb;
            tc_fence_after();
            const uint32_t kbase = smem_u32(sK + kr.buf * kTileBytes);
            const uint32_t d = tmem + sb * 128;
  #pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
              const uint64_t ad = sw128_kmajor_desc(smem_u32(sQ + kb * kSub));
              const uint64_t bd = sw128_kmajor_desc(kbase + kb * kSub);
  #pragma unroll
              for (int kq = 0; kq < 4; ++kq) tc_mma_bf16(d, ad + 2u * kq, bd + 2u * kq, IDESC, (kb | kq) ? 1u : 0u);
            }
            tc_commit(s_full(sb));
            tc_commit(k_empty(kr.buf));
            kr.next(kKst);
          }
          if (!ok) break;
          tc_commit(q_empty);  // every S of this unit is issued
          ++uc;
        }
        tc_commit(drain);
        drain_bar(drain, 0u, a.status);
      }
      __syncwarp();
    } else if (warp == 6) {
      if (lane == 0) {
        // ---- P V issuer: O += P_j V_j once the softmax threads have written P_j ----
        int uc = 0;
        int sb = 0;                          // buffer of the next P, in the S issuer's order
        Ring vr;
        uint32_t pph = 0;                    // bit b: phase of buffer b's next p_full wait
        bool ok = !(a.wait_limit_ns < kShortLimitNs) || wait_bar_wake(never, 0u, w);
        for (int k = 0; ok; ++k) {
          const int u = unit_of(k, b, G);
          if (u >= units) break;
          const AttnUnit t = decode(u, a);
          for (int j = 0; j < t.nk; ++j, sb = sb + 1 == kSbuf ? 0 : sb + 1) {
            // (for the unit's first key tile, also once the previous unit's O is read out)
            if (!wait_bar_wake(p_full(sb), (pph >> sb) & 1u, w) || (j == 0 && !wait_bar_wake(o_free, (uc & 1u) ^ 1u, w)) ||
                !wait_bar_wake(v_full(vr.buf), vr.phase, w)) {
              ok = false;
              break;
            }
            pph ^= 1u << sb;
            tc_fence_after();
            const uint32_t vbase = smem_u32(sV + vr.buf * kTileBytes);
            const uint32_t pa = tmem + sb * 128 + 64;  // P: the upper 64 columns, bf16 pairs
  #pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              // keys 16 kk ..: their 64-key half, then 2 KiB per 16 keys
              const uint64_t bd = sw128_mnmajor_desc(vbase + (kk >> 2) * kSub);
              tc_mma_bf16_tmem_a(tmem + kOcol, pa + 8u * kk, bd + 128u * (kk & 3), IDESC_PV, (j | kk) ? 1u : 0u);
            }
            tc_commit(s_free(sb));
            tc_commit(v_empty(vr.buf));
            vr.next(kVst);
            if (j + 1 == t.nk) tc_commit(o_full);
          }
          if (!ok) break;
          ++uc;
        }
        tc_commit(drain_pv);
        drain_bar(drain_pv, 0u, a.status);
      }
      __syncwarp();
    }
  } else if (warp < 4) {
    // ---- softmax: warps 0..3 (warp v reads TMEM lanes 32 v .. + 31) ----
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    const int row_in_tile = (warp & 3) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t ob = tmem + lane_base + kOcol;
    const float c = a.scale_log2;
    uint32_t sph = 0;                    // bit b: phase of buffer b's next s_full wait
    uint32_t uc = 0;                     // units done
    bool ok = true;
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool got = wait_bar_wake(bar, parity, w);
      return __all_sync(0xffffffffu, got);
    };
    int sbuf = 0, prev = kSbuf - 1;      // buffer of this key step and of the one before (one ring)
    for (int k = 0; ok; ++k) {
      const int u = unit_of(k, b, G);
      if (u >= units) break;
      const AttnUnit t = decode(u, a);
      const int row = t.mt * kTile + row_in_tile;
      float m_used = -INFINITY, l_run = 0.f;
      for (int j = 0; j < t.nk; ++j, prev = sbuf, sbuf = sbuf + 1 == kSbuf ? 0 : sbuf + 1) {
        const uint32_t sb = tmem + lane_base + sbuf * 128;
        if (!wait_all(s_full(sbuf), (sph >> sbuf) & 1u)) {
          ok = false;
          break;
        }
        sph ^= 1u << sbuf;
        tc_fence_after();
        // allowed keys of this tile: key0 + i for i <= kmax (causal: key <= row; always key < M)
        const int key0 = key_tile(k, t, j) * kTile;
        int kmax = a.M - 1 - key0;
        if (a.causal && row - key0 < kmax) kmax = row - key0;
        const bool masked = kmax < kTile - 1;
        // every key tile a row visits holds at least one allowed key (its own, or key < M)
        if (!TP_CHECK(kmax >= 0, a.status)) kmax = 0;
        // the whole row of S_j (128 scores) in registers: its maximum, then the weights
        uint32_t s[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(sb + cc * 32, s[cc]);
        tmem_ld_wait();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_reg_fence(s[cc]);
        if (masked) {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (cc * 32 + i > kmax) s[cc][i] = __float_as_uint(-INFINITY);
        }
        // P = 2^(t - m) as bf16 pairs over the upper 64 columns of the S buffer: keys 64 hh ..
        // 64 hh + 63 into columns 64 + 32 hh (the scores are all in registers by now).  The
        // row sum adds the float32 weights before their rounding to bf16 for the P V product;
        // the roundings (2^-9 relative each, independent) move an output by far less than its
        // own bf16 rounding.  Paired float32 operations: two scores per FFMA2 and FADD2.
        // Returns the row sum; with `watch`, also the largest exponent argument t - m (targ).
        auto make_p = [&](float m_sh, bool watch, float &targ) -> float {
          float2 sum4[4];
          float tm4[4];
#pragma unroll
          for (int g4 = 0; g4 < 4; ++g4) {
            sum4[g4] = make_float2(0.f, 0.f);
            tm4[g4] = -INFINITY;
          }
          const float2 c2 = make_float2(c, c), nm2 = make_float2(-m_sh, -m_sh);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const uint32_t *v = s[2 * hh + (i >> 4)];
              const float2 t2 = __ffma2_rn(
                  make_float2(__uint_as_float(v[(2 * i) & 31]), __uint_as_float(v[(2 * i + 1) & 31])), c2, nm2);
              if (watch) tm4[i & 3] = fmax3(tm4[i & 3], t2.x, t2.y);
              const float2 e = make_float2(ex2_approx(t2.x), ex2_approx(t2.y));
              pk[i] = pack_bf16x2(e.x, e.y);
              sum4[i & 3] = __fadd2_rn(sum4[i & 3], e);
            }
            tmem_st32(sb + 64 + hh * 32, pk);
          }
          targ = fmaxf(fmaxf(tm4[0], tm4[1]), fmaxf(tm4[2], tm4[3]));
          return ((sum4[0].x + sum4[0].y) + (sum4[1].x + sum4[1].y)) +
                 ((sum4[2].x + sum4[2].y) + (sum4[3].x + sum4[3].y));
        };
        // The unit's first key tile sets the shift from the tile's maximum.  A later tile first
        // makes P against the current shift, watching the largest exponent argument alongside
        // (its maxima run on the ALU beside the exponentials on the XU); only where some score
        // would exceed 2^8 is the tile made again from its maximum, as the first one is (lanes
        // whose shift stays then make the same P again).
        float sum = 0.f, alpha = 1.0f, m_new = m_used, targ = 0.f;
        bool raise = false;
        bool redo = j == 0;
        if (!redo) {
          sum = make_p(m_used, true, targ);
          redo = __any_sync(0xffffffffu, targ > kRescaleGap);
        }
        if (redo) {
          // row maximum: sixteen chains of four three-input maxima over 8 scores each, then a tree
          float m16[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const uint32_t *v = s[q >> 2] + (q & 3) * 8;
            float m = fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
            m = fmax3(m, __uint_as_float(v[3]), __uint_as_float(v[4]));
            m = fmax3(m, __uint_as_float(v[5]), __uint_as_float(v[6]));
            m16[q] = fmaxf(m, __uint_as_float(v[7]));
          }
          float m6[6];
#pragma unroll
          for (int q = 0; q < 5; ++q) m6[q] = fmax3(m16[3 * q], m16[3 * q + 1], m16[3 * q + 2]);
          m6[5] = m16[15];
          const float mx = fmaxf(fmax3(m6[0], m6[1], m6[2]), fmax3(m6[3], m6[4], m6[5]));
          const float m_tile = mx * c;
          raise = m_tile > m_used + kRescaleGap;
          m_new = raise ? m_tile : m_used;
          alpha = raise ? ex2_approx(m_used - m_new) : 1.0f;  // 0 on the first tile
          sum = make_p(m_new, false, targ);
        }
        l_run = fmaf(l_run, alpha, sum);
        // A raised shift also scales the accumulated O, once every P V issued before this step
        // is complete.  The last of them, P_{j-1} V_{j-1}, completes the phase of
        // s_free(buffer of j - 1) whose parity is that of the s_full phase step j - 1 waited on.
        // That barrier's previous phase is complete already (S_{j-1} was issued after it), and
        // its next one needs P_{j+2}, which this step precedes: the parity names one phase.
        if (j > 0 && __any_sync(0xffffffffu, raise)) {
          if (!wait_all(s_free(prev), ((sph >> prev) & 1u) ^ 1u)) {
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
        m_used = m_new;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full(sbuf));
      }
      if (!ok) break;
      // the row sum to the output warps, through slot uc % 2 (once they have read that slot's
      // sum of two units before: a fresh barrier's previous phase counts as complete)
      const uint32_t par = uc & 1u;
      if (!wait_all(l_empty(par), ((uc >> 1) & 1u) ^ 1u)) break;
      l_buf[par * 128 + row_in_tile] = l_run;
      mbar_arrive(l_full(par));
      ++uc;
    }
  } else if (warp >= 8) {
    // ---- output: warps 8..11 (warp v reads TMEM lanes 32 (v % 4) .. + 31) ----
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOut));
    const int row_in_tile = (warp & 3) * 32 + lane;
    const uint32_t ob = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kOcol;
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool got = wait_bar_wake(bar, parity, w);
      return __all_sync(0xffffffffu, got);
    };
    uint32_t uc = 0;  // units read out
    for (int k = 0;; ++k) {
      const int u = unit_of(k, b, G);
      if (u >= units) break;
      const AttnUnit t = decode(u, a);
      const int row = t.mt * kTile + row_in_tile;
      const uint32_t par = uc & 1u;
      if (!wait_all(o_full, uc & 1u) || !wait_all(l_full(par), (uc >> 1) & 1u)) break;
      tc_fence_after();
      const float inv = 1.0f / l_buf[par * 128 + row_in_tile];
      mbar_arrive(l_empty(par));
      const bool in_row = TP_CHECK((t.head + 1) * static_cast<long long>(kAttnHeadDim) <= a.ldo, a.status);
      __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(a.O) + static_cast<long long>(row) * a.ldo +
                            static_cast<long long>(t.head) * kAttnHeadDim;
      uint4 *dst = reinterpret_cast<uint4 *>(orow);
      // 32-byte stores (whole sectors) where the row is 32-byte aligned, else 16-byte ones
      const bool wide = (reinterpret_cast<uintptr_t>(orow) & 31u) == 0;
      // the row of O / l as bf16 pairs (64 registers), a chunk of 32 columns at a time; then O is
      // free for the next unit's first P V, and the stores follow
      uint32_t p[64];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t r[32];
        tmem_ld32(ob + cc * 32, r);
        tmem_ld_wait();
        tmem_reg_fence(r);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          p[16 * cc + i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
      }
      tc_fence_before();
      mbar_arrive(o_free);
      if (row < a.M && in_row) {
        if (wide) {
#pragma unroll
          for (int q = 0; q < 8; ++q) st_global_v8(orow + 16 * q, p + 8 * q);
        } else {
#pragma unroll
          for (int g4 = 0; g4 < 16; ++g4) dst[g4] = make_uint4(p[4 * g4], p[4 * g4 + 1], p[4 * g4 + 2], p[4 * g4 + 3]);
        }
      }
      ++uc;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int attention_key_box_rows() { return kTile; }

cudaError_t launch_attention(const CUtensorMap &mapQ, const CUtensorMap &mapK, const CUtensorMap &mapV,
                             const AttnArgs &args, int num_sms, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const long long units = static_cast<long long>(args.heads) * args.m_tiles;
  if (units <= 0) return cudaSuccess;
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  // launched as a programmatic dependent of the previous kernel (the QKV projection)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_fwd_kernel, mapQ, mapK, mapV, args);
}

}  // namespace tp
