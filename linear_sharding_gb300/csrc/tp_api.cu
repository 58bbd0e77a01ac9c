// tp_api.cu - the C ABI of libtpmlp.so (declared in include/tp_mlp.h):
// argument checks, the shard handles, TMA tensor maps, the per-shape launch
// plan and the order of the kernels of one forward pass.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <new>

#include "tp_internal.h"

using namespace tp;

struct tp_shards {
  int kind = 0;  // 0 = MLP, 1 = QKV
  int device = 0;
  int64_t H = 0, F = 0, Fs = 0;  // QKV: F = H, Fs = W (head columns per shard)
  int T = 0;
  tp_act_t act = TP_ACT_GELU_ERF;
  tp_dtype_t dt = TP_BF16;
  int n_heads = 0, head_dim = 0;
  int64_t R1 = 0;  // packed first-layer rows per shard (Fs, 2 Fs for SwiGLU, 3 W for QKV)
  // Packed shards: logically W1_i^T [T][R1][H] and W2_i^T [T][H][Fs] (K-major).
  // Float32: stored so.  Bfloat16: in k-tiles of 64, [H/64][T R1][64] and
  // [T][Fs/64][H][64], so that every 128-row x 64 copy the GEMMs make of a
  // weight is one contiguous 16 KiB block.
  void *w1p = nullptr;
  void *w2p = nullptr;
  int bn1 = 256, bn2 = 256;
  CUtensorMap map_w1_b, map_w1_a, map_w2_b, map_w2_a;
  // backward operands: W1 [H x ncols] and W2 [F x H] in the caller's layout
  bool backward = false;
  void *w1o = nullptr, *w2o = nullptr;
  int bn_dh = 256;  // tile width of dH = dZ W2^T (its N is F, tiles stay inside a shard)
  CUtensorMap map_w2o_bn, map_w2o_128, map_w1o_bn, map_w1o_128;
};

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxShards = 64;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
constexpr int kDecodeMaxM = 16;

struct DevState {
  bool ready = false;
  int sms = 0;
  unsigned int *status = nullptr;
  // Dense bf16 tensor flop per byte of HBM traffic from the device's own
  // figures (peak SM clock, memory clock and bus width): the exchange rate
  // the planners use between GEMM work and float32 partial traffic.
  double queried_balance = 0.0;
};

std::mutex g_mu;
DevState g_dev[kMaxDevices];
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};
// tp_set_machine_balance: a caller's measured flop-per-byte figure (0: use
// the queried one).
std::atomic<double> g_balance_override{0.0};
// tp_set_rowpar_schedule: whether the row-parallel GEMM may use the wide tiles.
std::atomic<int> g_rowpar_wide{1};

// Dense bf16 tensor-core flop per SM per clock (tcgen05.mma, kind::f16):
// a 128 x 256 x 16 MMA every 128 cycles.
constexpr double kFlopPerSmClock = 8192.0;

// Failure injection (tp_inject_alloc_failures): device allocations still to fail.
std::atomic<int> g_fail_allocs{0};

bool take_injected_failure() {
  int n = g_fail_allocs.load();
  while (n > 0)
    if (g_fail_allocs.compare_exchange_weak(n, n - 1)) return true;
  return false;
}

// Every device allocation of the library goes through these two.
cudaError_t lib_malloc(void **p, size_t bytes) {
  if (take_injected_failure()) return cudaErrorMemoryAllocation;
  return cudaMalloc(p, bytes);
}

cudaError_t lib_malloc_async(void **p, size_t bytes, cudaStream_t st) {
  if (take_injected_failure()) return cudaErrorMemoryAllocation;
  return cudaMallocAsync(p, bytes, st);
}

tp_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return TP_OK;
  if (e == cudaErrorMemoryAllocation) return TP_ERR_OOM;
  return TP_ERR_CUDA;
}

#define TP_TRY(expr)                      \
  do {                                    \
    const tp_status_t _st = (expr);       \
    if (_st != TP_OK) return _st;         \
  } while (0)

#define TP_CUDA(expr) TP_TRY(cuda_status(expr))

// Per-device state: SM count and the status word, created on first use.
tp_status_t dev_state(DevState **out, int *dev_out = nullptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TP_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DevState &d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return TP_ERR_CUDA;
    if (major != 10 || minor != 3) return TP_ERR_ARCH;
    int clk_khz = 0, mem_khz = 0, bus_bits = 0;
    cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, dev);
    cudaDeviceGetAttribute(&mem_khz, cudaDevAttrMemoryClockRate, dev);
    cudaDeviceGetAttribute(&bus_bits, cudaDevAttrGlobalMemoryBusWidth, dev);
    // Double data rate: two transfers of bus_bits per memory clock.
    const double flops = kFlopPerSmClock * sms * clk_khz * 1e3;
    const double bytes = 2.0 * mem_khz * 1e3 * bus_bits / 8.0;
    d.queried_balance = (flops > 0.0 && bytes > 0.0) ? flops / bytes : 300.0;
    unsigned int *st = nullptr;
    if (lib_malloc(reinterpret_cast<void **>(&st), 256) != cudaSuccess) return TP_ERR_OOM;
    if (cudaMemset(st, 0, 256) != cudaSuccess) {
      cudaFree(st);
      return TP_ERR_CUDA;
    }
    d.sms = sms;
    d.status = st;
    d.ready = true;
  }
  *out = &d;
  if (dev_out) *dev_out = dev;
  return TP_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D bf16 tensor map, dims {d0 (contiguous), d1, d2}, byte strides {s1, s2},
// box {64, box1, 1}, 128-byte swizzle, zero fill out of bounds.
tp_status_t make_map(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                     uint64_t s1, uint64_t s2, uint32_t box1) {
  EncodeTiledFn f = encode_fn();
  if (!f) return TP_ERR_CUDA;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {64, box1, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                       strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TP_OK : TP_ERR_CUDA;
}

// 4-D bf16 tensor map of an MN-major GEMM operand stored [segs][K][mn] (mn
// elements per segment, a multiple of 64): dims {64, K, mn / 64, segs}, byte
// strides {mn x 2, 128, K x mn x 2}, box {64, 64, kMnPairBox, 1}, 128-byte
// swizzle, zero fill past K.  See kMnPairBox.
tp_status_t make_map_mn_pairs(CUtensorMap *m, const void *base, uint64_t mn, uint64_t K, uint64_t segs) {
  EncodeTiledFn f = encode_fn();
  if (!f) return TP_ERR_CUDA;
  const cuuint64_t dims[4] = {64, K, mn / 64, segs};
  const cuuint64_t strides[3] = {mn * 2, 128, K * mn * 2};
  const cuuint32_t box[4] = {64, 64, static_cast<cuuint32_t>(kMnPairBox), 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TP_OK : TP_ERR_CUDA;
}

// Tensor maps of the k-tile-blocked bf16 weights (operand mode kKtileBlocked:
// coordinate (0, row, k-tile)).  W1: k-tile kt of all T R1 rows; W2: k-tile
// kt of shard i is plane i (Ks/64) + kt of H rows.  Ks is the per-shard K of W2.
tp_status_t make_weight_maps(tp_shards *s, int64_t Ks) {
  const int64_t rows1 = s->T * s->R1, kt1 = s->H / 64, kt2 = s->T * (Ks / 64);
  tp_status_t r = make_map(&s->map_w1_b, s->w1p, 64, rows1, kt1, 128, rows1 * 128, s->bn1);
  if (r == TP_OK) r = make_map(&s->map_w1_a, s->w1p, 64, rows1, kt1, 128, rows1 * 128, 128);
  if (r == TP_OK) r = make_map(&s->map_w2_b, s->w2p, 64, s->H, kt2, 128, s->H * 128, s->bn2);
  if (r == TP_OK) r = make_map(&s->map_w2_a, s->w2p, 64, s->H, kt2, 128, s->H * 128, 128);
  return r;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool ranges_overlap(const void *a, size_t abytes, const void *b, size_t bbytes) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bbytes && b0 < a0 + abytes;
}

size_t esize(tp_dtype_t dt) { return dt == TP_BF16 ? 2 : 4; }

size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Cost of one byte of float32 partials (written once, read by the
// shard-sum) in k-tiles of a 128 x bn tensor-core tile: the machine balance
// (flop per HBM byte) over the flop of one k-tile.
double ktile_per_partial_byte(const DevState *d, int bn) {
  const double o = g_balance_override.load();
  const double balance = o > 0.0 ? o : d->queried_balance;
  return balance / (2.0 * 128.0 * bn * 64.0);
}

GemmArgs base_args(const DevState *d) {
  GemmArgs g;
  std::memset(&g, 0, sizeof g);
  g.group_m = 16;
  g.status = d->status;
  g.wait_limit_ns = g_wait_ns.load();
  return g;
}

// ---- planning ---------------------------------------------------------------

// Number of accumulation slots of a row-parallel GEMM with `tiles` output
// tiles of `kt_total` k-tiles, split into slots that each cover whole shard
// groups (divisors of T) or, when `sub_ok`, also sub-ranges of a shard.
// Cost = waves x k-tiles per unit (compute or weight streaming) plus the
// float32 partial traffic (written once, read by the shard-sum) expressed in
// k-tile units.
int choose_slots(int64_t tiles, int T, int kt_per_seg, int sms, double ktile_per_partial_byte,
                 int64_t partial_bytes, bool sub_ok, int max_slots = 1 << 30) {
  int best = 1;
  double best_cost = 1e300;
  auto consider = [&](int S) {
    const int64_t kt_total = static_cast<int64_t>(T) * kt_per_seg;
    if (kt_total % S || S > max_slots) return;
    const int64_t units = tiles * S;
    const int64_t waves = cdiv(units, sms);
    double cost = static_cast<double>(waves) * static_cast<double>(kt_total / S);
    if (S > 1) cost += ktile_per_partial_byte * static_cast<double>(partial_bytes) * (2.0 * S + 1.0) / sms;
    if (cost < best_cost * 0.999) {
      best_cost = cost;
      best = S;
    }
  };
  for (int S = 1; S <= T; ++S)
    if (T % S == 0) consider(S);
  if (sub_ok)
    for (int sub = 2; sub <= 8; ++sub)
      if (kt_per_seg % sub == 0 && T * sub <= kMaxShards) consider(T * sub);
  return best;
}

struct MlpPlan {
  bool simt = false, decode = false;
  int slots1 = 1;  // decode: split-K slots of the first layer
  int slots2 = 1;  // second layer accumulation slots (1 = all shards in one accumulator)
  size_t y_bytes = 0;    // Y, T x M x Fs elements
  size_t col_bytes = 0;  // first-layer scratch (decode split-K partials)
  size_t row_bytes = 0;  // second-layer scratch (float32 partials)
  size_t total() const { return round256(y_bytes) + round256(col_bytes) + round256(row_bytes); }
};

// budget > 0 (AUTO only): when the AUTO plan's workspace exceeds `budget` bytes, refit it: no
// second-layer partials (all shards in one TMEM accumulator) and, for decode, as many first-layer
// split-K slots as fit.  A plan that fits is left as it is.
tp_status_t plan_mlp(const tp_shards *s, int64_t M, tp_variant_t v, const DevState *d, MlpPlan *p,
                     size_t budget = 0) {
  *p = MlpPlan();
  const int sms = d->sms;
  const double per_byte_tc = ktile_per_partial_byte(d, s->bn2);
  const int64_t H = s->H, Fs = s->Fs, T = s->T, R1 = s->R1;
  const size_t eb = esize(s->dt);
  p->y_bytes = static_cast<size_t>(T * M * Fs) * eb;
  if (s->dt == TP_F32) {
    p->simt = true;
    p->slots2 = (v == TP_VAR_PARTIALS) ? static_cast<int>(T) : 1;
  } else if (M <= kDecodeMaxM) {
    p->decode = true;
    const int kps = static_cast<int>(Fs / 64);
    // Weight streaming: one 128 x 64 bf16 A tile (16 KiB) per k-tile.
    const double per_byte = 1.0 / (128.0 * 64.0 * 2.0);
    p->slots1 = choose_slots((T * R1) / 128, 1, static_cast<int>(H / 64), sms, per_byte,
                             static_cast<int64_t>(M * T * R1 * 4), true);
    if (v == TP_VAR_TMEM_ACC)
      p->slots2 = 1;
    else if (v == TP_VAR_PARTIALS)
      p->slots2 = static_cast<int>(T);
    else
      p->slots2 = choose_slots(H / 128, static_cast<int>(T), kps, sms, per_byte,
                               static_cast<int64_t>(M * H * 4), true);
    p->col_bytes = static_cast<size_t>(p->slots1 * M * T * R1) * 4;
  } else {
    const int kps = static_cast<int>(Fs / 64);
    if (v == TP_VAR_TMEM_ACC)
      p->slots2 = 1;
    else if (v == TP_VAR_PARTIALS)
      p->slots2 = static_cast<int>(T);
    else {
      // Tensor-bound: one k-tile of a 128 x bn2 tile is 2*128*bn2*64 flop; a
      // partial byte costs the machine balance in flop.
      p->slots2 = choose_slots(cdiv(M, 128) * (H / s->bn2), static_cast<int>(T), kps, sms, per_byte_tc,
                               static_cast<int64_t>(M * H * 4), false);
    }
  }
  p->row_bytes = p->slots2 > 1 ? static_cast<size_t>(p->slots2 * M * H) * 4 : 0;
  if (budget > 0 && v == TP_VAR_AUTO && p->total() > budget) {
    p->slots2 = 1;
    p->row_bytes = 0;
    if (p->decode) {
      const size_t per_slot = static_cast<size_t>(M * T * R1) * 4;
      const size_t fixed = round256(p->y_bytes) + 255;
      const int64_t fit = budget > fixed ? static_cast<int64_t>((budget - fixed) / per_slot) : 0;
      const int cap = static_cast<int>(fit < 1 ? 1 : (fit > p->slots1 ? p->slots1 : fit));
      p->slots1 = choose_slots((T * R1) / 128, 1, static_cast<int>(H / 64), sms, 1.0 / (128.0 * 64.0 * 2.0),
                               static_cast<int64_t>(M * T * R1 * 4), true, cap);
      p->col_bytes = static_cast<size_t>(p->slots1) * per_slot;
    }
  }
  return TP_OK;
}

// ---- forward passes ---------------------------------------------------------

Epi act_epi(tp_act_t act) {
  return act == TP_ACT_GELU_ERF ? EPI_GELU_BF16 : act == TP_ACT_SWIGLU ? EPI_SWIGLU_BF16 : EPI_IDENT_BF16;
}

GemmCfg cfg_for(int bn) { return bn == 256 ? CFG_N256 : CFG_N128; }

// 256-wide tiles over more than one 128-row block of tokens run on CTA pairs
// (cta_group::2): half the B-tile traffic per SM and a deeper stage ring.
bool use_pair(int bn, int64_t M) { return bn == 256 && M > 128; }

// A residual added to a row-parallel layer's output Z [M x H]: Z += add_f32 (float32)
// and/or Z += add_bf16 (bf16), then, with out_bf16, out_bf16 = bf16(Z).  All null: none.
struct Residual {
  const float *add_f32 = nullptr;
  const void *add_bf16 = nullptr;
  void *out_bf16 = nullptr;
  bool any() const { return add_f32 || add_bf16 || out_bf16; }
};

// The residual as separate elementwise kernels over Z (when it is not fused).
tp_status_t apply_residual(const DevState *d, float *Z, int64_t n, const Residual &r, cudaStream_t st) {
  if (r.add_bf16 || r.out_bf16) {
    if (!r.add_bf16 || !r.out_bf16) return TP_ERR_ARG;
    TP_CUDA(launch_residual(r.add_bf16, Z, Z, r.out_bf16, n, d->sms, st));
  }
  if (r.add_f32) TP_CUDA(launch_add_inplace(Z, r.add_f32, n, d->sms, st));
  return TP_OK;
}

// Wide schedule of a row-parallel CTA-pair GEMM with one accumulation slot (launch_gemm_wide):
// each of the m_tiles 256-row blocks of H columns is cut into q tiles whose widths are multiples
// of 32 that differ by at most 32 (nb of bn columns, q - nb of bn - 32), every tile wider than 256
// columns (two MMAs per k-step into two accumulators) and at most kWideMaxN, in one or two rounds
// of the clusters, q as large as that allows.  A cluster's single accumulator of up to
// kWideMaxN columns is drained before its next tile starts, so each round after the first
// exposes one epilogue, priced as epi_ktiles k-tiles of a 480-column tile: 6 for the float32
// output, 24 where the epilogue also reads a residual and writes its bf16 copy (timed on one
// GPU: the block's O-projection, 64 k-tiles at M = 4096, ran faster on 256-column tiles and its
// MLP down-projection, 256 k-tiles, on the wide ones; the float32 O-projection alone, on the
// wide ones).  Against the 256-column tiles
// in rounds (their epilogues hidden behind the next tile), with the tensor-pipe activity
// measured for each form at this size (about 90 % and 80 %), priced in column-k-tiles.  kt: the
// k-tiles of one tile.  bn = 0: the 256-column tiles.  At M = 2048, H = 4096 on 76 clusters:
// 128 tiles of 256 columns take two rounds, 8 x 9 tiles of 480 and 448 columns one.
struct WidePlan {
  int bn = 0, nb = 0, q = 0;
};
constexpr double kEpiKtilesF32 = 6.0, kEpiKtilesResid = 24.0;
WidePlan plan_wide(int m_tiles, int64_t H, int clusters, int64_t kt, double epi_ktiles = kEpiKtilesF32) {
  WidePlan best;
  if (m_tiles < 1 || H % 256 != 0 || clusters < m_tiles || kt < 1) return best;
  const int64_t units = H / 32;  // 32-column units of a row block
  const int64_t rounds_u = cdiv(static_cast<int64_t>(m_tiles) * (H / 256), clusters);
  const double cost_u = static_cast<double>(rounds_u) * 256.0 * kt / 0.80;
  double best_cost = 0.95 * cost_u;  // the wide tiles must win by 5 %
  for (int rounds = 1; rounds <= 2; ++rounds) {
    for (int64_t q = rounds * clusters / m_tiles; q >= 1; --q) {
      const int64_t w1 = cdiv(units, q);        // widest tile, in units
      const int64_t nb = units - q * (w1 - 1);  // tiles of w1 units; the others have w1 - 1
      const int64_t narrowest = nb == q ? w1 : w1 - 1;
      if (32 * narrowest <= 256) continue;      // a tile this narrow has one MMA: fewer, wider tiles
      if (32 * w1 > kWideMaxN) break;           // fewer tiles would only be wider
      const int64_t rounds_w = cdiv(static_cast<int64_t>(m_tiles) * q, clusters);
      const double cost = static_cast<double>(rounds_w) * 32.0 * w1 * kt / 0.90 + (rounds_w - 1) * epi_ktiles * 480.0;
      if (cost < best_cost) {
        best_cost = cost;
        best.bn = static_cast<int>(32 * w1);
        best.nb = static_cast<int>(nb);
        best.q = static_cast<int>(q);
      }
      break;
    }
  }
  return best;
}

// A B operand's 3-D tensor as make_map takes it (base, dims, byte strides), for tensor maps of
// other box heights over it.
struct BTensor {
  const void *base;
  uint64_t d0, d1, d2, s1, s2;
};

// Launch a CTA-pair GEMM with float32 output and one slot (epi EPI_F32 or EPI_F32_RESID; its
// output columns N along B's rows) on the wide schedule when plan_wide has one and
// tp_set_rowpar_schedule allows it; *done says whether it ran.  b128: the B map with the
// 128-row box, over `bt`.
tp_status_t try_wide(const DevState *d, Epi epi, const GemmArgs &g, int64_t N, const CUtensorMap &mapA,
                     const CUtensorMap &b128, const BTensor &bt, cudaStream_t st, bool *done) {
  *done = false;
  if (g_rowpar_wide.load() == 0) return TP_OK;
  const WidePlan wp = plan_wide(g.m_tiles, N, d->sms / 2, g.kt_total,
                                epi == EPI_F32_RESID ? kEpiKtilesResid : kEpiKtilesF32);
  if (wp.bn == 0) return TP_OK;
  // the same tensor with the row counts of the tiles' second B pieces as boxes
  CUtensorMap mb2, mbr;
  TP_TRY(make_map(&mb2, bt.base, bt.d0, bt.d1, bt.d2, bt.s1, bt.s2, static_cast<uint32_t>(wp.bn - 256) / 2));
  if (wp.nb < wp.q)
    TP_TRY(make_map(&mbr, bt.base, bt.d0, bt.d1, bt.d2, bt.s1, bt.s2, static_cast<uint32_t>(wp.bn - 288) / 2));
  else
    mbr = mb2;
  GemmArgs gw = g;
  gw.wide_bn = wp.bn;
  gw.wide_nb = wp.nb;
  gw.wide_q = wp.q;
  TP_CUDA(launch_gemm_wide(epi, mapA, b128, mb2, mbr, gw, d->sms, st));
  *done = true;
  return TP_OK;
}

// Row-parallel GEMM over T shards into Z, with `slots` accumulation slots
// (slots > 1: float32 partials in P, then the shard-sum).  A residual is fused
// into the GEMM's epilogue with one slot, and applied after the shard-sum otherwise.
tp_status_t rowpar_tc(const tp_shards *s, const DevState *d, const CUtensorMap &mapA, int a_seg,
                      int64_t M, int slots, float *P, float *Z, cudaStream_t st, const Residual &res = Residual()) {
  const int64_t H = s->H;
  const bool pair = use_pair(s->bn2, M);
  GemmArgs g = base_args(d);
  g.m_tiles = static_cast<int>(cdiv(M, pair ? 256 : 128));
  g.n_tiles = static_cast<int>(H / s->bn2);
  g.slots = slots;
  g.kt_per_seg = static_cast<int>(s->Fs / 64);
  g.kt_total = s->T * g.kt_per_seg;
  g.kt_per_slot = g.kt_total / slots;
  g.a_seg = a_seg;
  g.b_seg = kKtileBlocked;
  g.rows_valid = static_cast<int>(M);
  g.cols_valid = static_cast<int>(H);
  g.out = slots > 1 ? static_cast<void *>(P) : static_cast<void *>(Z);
  g.ld_out = H;
  g.slot_stride = M * H;
  Epi epi = EPI_F32;
  if (slots == 1 && res.any()) {
    epi = EPI_F32_RESID;
    g.aux = res.add_f32;
    g.aux2 = res.add_bf16;
    g.out2 = res.out_bf16;
  }
  bool done = false;
  if (pair && slots == 1)
    TP_TRY(try_wide(d, epi, g, H, mapA, s->map_w2_a, BTensor{s->w2p, 64, static_cast<uint64_t>(H),
                                                       static_cast<uint64_t>(g.kt_total), 128,
                                                       static_cast<uint64_t>(H) * 128},
                    st, &done));
  if (!done && pair)
    TP_CUDA(launch_gemm(CFG_PAIR_N256, epi, mapA, s->map_w2_a, g, d->sms, st));
  else if (!done)
    TP_CUDA(launch_gemm(cfg_for(s->bn2), epi, mapA, s->map_w2_b, g, d->sms, st));
  if (slots > 1) {
    TP_CUDA(launch_shard_sum_strided(P, slots, M * H, M * H, Z, d->sms, st));
    TP_TRY(apply_residual(d, Z, M * H, res, st));
  }
  return TP_OK;
}

// Column-parallel GEMM of all shards: out[shard][M][shard_cols] bf16.
tp_status_t colpar_tc(const tp_shards *s, const DevState *d, const void *X, int64_t M, Epi epi,
                      void *out, int64_t shard_cols, cudaStream_t st) {
  const int64_t H = s->H;
  CUtensorMap mx;
  TP_TRY(make_map(&mx, X, H, M, 1, H * 2, M * H * 2, 128));
  const bool pair = use_pair(s->bn1, M);
  GemmArgs g = base_args(d);
  g.m_tiles = static_cast<int>(cdiv(M, pair ? 256 : 128));
  g.n_tiles = static_cast<int>(s->T * s->R1 / s->bn1);
  g.slots = 1;
  g.b_seg = kKtileBlocked;
  g.kt_total = static_cast<int>(H / 64);
  g.kt_per_seg = g.kt_total;
  g.kt_per_slot = g.kt_total;
  g.rows_valid = static_cast<int>(M);
  g.cols_valid = static_cast<int>(s->T * shard_cols);
  g.out = out;
  g.ld_out = shard_cols;
  g.shard_stride = M * shard_cols;
  g.shard_cols = static_cast<int>(shard_cols);
  if (pair)
    TP_CUDA(launch_gemm(CFG_PAIR_N256, epi, mx, s->map_w1_a, g, d->sms, st));
  else
    TP_CUDA(launch_gemm(cfg_for(s->bn1), epi, mx, s->map_w1_b, g, d->sms, st));
  return TP_OK;
}

// Decode first layer: operands swapped (weight rows x tokens), split-K
// float32 partials P1, then the activation into Y.
tp_status_t colpar_decode(const tp_shards *s, const DevState *d, const MlpPlan &p, const void *X,
                          int64_t M, tp_act_t act, void *Y, float *P1, cudaStream_t st) {
  const int64_t H = s->H, T = s->T, Fs = s->Fs, rows1 = T * s->R1;
  CUtensorMap mxb;
  TP_TRY(make_map(&mxb, X, H, M, 1, H * 2, M * H * 2, 16));
  GemmArgs g = base_args(d);
  g.m_tiles = static_cast<int>(rows1 / 128);
  g.n_tiles = 1;
  g.slots = p.slots1;
  g.a_seg = kKtileBlocked;
  g.kt_total = static_cast<int>(H / 64);
  g.kt_per_seg = g.kt_total;
  g.kt_per_slot = g.kt_total / p.slots1;
  g.group_m = 1;
  g.rows_valid = static_cast<int>(rows1);
  g.cols_valid = static_cast<int>(M);
  g.out = P1;
  g.ld_out = rows1;
  g.slot_stride = M * rows1;
  TP_CUDA(launch_gemm(CFG_N16, EPI_F32_T, s->map_w1_a, mxb, g, d->sms, st));
  TP_CUDA(launch_decode_act(P1, p.slots1, M * rows1, rows1, static_cast<int>(M), static_cast<int>(T),
                            static_cast<int>(Fs), act, act == TP_ACT_SWIGLU, Y, st));
  return TP_OK;
}

// Decode second layer: W2 rows x tokens, per-shard (and split) slots, then
// the shard-sum.
tp_status_t rowpar_decode(const tp_shards *s, const DevState *d, const MlpPlan &p, const void *Y,
                          int64_t M, float *Z, float *P2, cudaStream_t st) {
  const int64_t H = s->H, T = s->T, Fs = s->Fs;
  CUtensorMap myb;
  TP_TRY(make_map(&myb, Y, Fs, M, T, Fs * 2, M * Fs * 2, 16));
  GemmArgs g = base_args(d);
  g.m_tiles = static_cast<int>(H / 128);
  g.n_tiles = 1;
  g.slots = p.slots2;
  g.kt_per_seg = static_cast<int>(Fs / 64);
  g.kt_total = static_cast<int>(T) * g.kt_per_seg;
  g.kt_per_slot = g.kt_total / p.slots2;
  g.a_seg = kKtileBlocked;
  g.b_seg = 1;
  g.group_m = 1;
  g.rows_valid = static_cast<int>(H);
  g.cols_valid = static_cast<int>(M);
  g.out = p.slots2 > 1 ? static_cast<void *>(P2) : static_cast<void *>(Z);
  g.ld_out = H;
  g.slot_stride = M * H;
  TP_CUDA(launch_gemm(CFG_N16, EPI_F32_T, s->map_w2_a, myb, g, d->sms, st));
  if (p.slots2 > 1) TP_CUDA(launch_shard_sum_strided(P2, p.slots2, M * H, M * H, Z, d->sms, st));
  return TP_OK;
}

tp_status_t colpar_simt(const tp_shards *s, const void *X, int64_t M, tp_act_t act, void *Y,
                        cudaStream_t st) {
  const int64_t H = s->H, T = s->T, Fs = s->Fs;
  SimtArgs a;
  std::memset(&a, 0, sizeof a);
  a.A = static_cast<const float *>(X);
  a.B = static_cast<const float *>(s->w1p);
  a.lda = H;
  a.ldb = H;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(T * s->R1);
  a.k_seg = static_cast<int>(H);
  a.nseg = 1;
  a.segs_per_slot = 1;
  a.epi = act_epi(act);
  a.out = static_cast<float *>(Y);
  a.ld_out = Fs;
  a.shard_stride = M * Fs;
  a.shard_cols = static_cast<int>(Fs);
  TP_CUDA(launch_simt_gemm(a, st));
  return TP_OK;
}

tp_status_t rowpar_simt(const tp_shards *s, const DevState *d, const MlpPlan &p, const void *Y,
                        int64_t M, float *Z, float *P, cudaStream_t st) {
  const int64_t H = s->H, T = s->T, Fs = s->Fs;
  SimtArgs a;
  std::memset(&a, 0, sizeof a);
  a.A = static_cast<const float *>(Y);
  a.B = static_cast<const float *>(s->w2p);
  a.lda = Fs;
  a.ldb = Fs;
  a.a_seg = M * Fs;
  a.b_seg = H * Fs;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(H);
  a.k_seg = static_cast<int>(Fs);
  a.nseg = static_cast<int>(T);
  a.segs_per_slot = p.slots2 > 1 ? static_cast<int>(T) / p.slots2 : static_cast<int>(T);
  a.epi = EPI_F32;
  a.out = p.slots2 > 1 ? P : Z;
  a.ld_out = H;
  a.slot_stride = M * H;
  TP_CUDA(launch_simt_gemm(a, st));
  if (p.slots2 > 1) TP_CUDA(launch_shard_sum_strided(P, p.slots2, M * H, M * H, Z, d->sms, st));
  return TP_OK;
}

tp_status_t colpar_any(const tp_shards *s, const DevState *d, const MlpPlan &p, const void *X,
                       int64_t M, tp_act_t act, void *Y, char *ws_col, cudaStream_t st) {
  if (p.simt) return colpar_simt(s, X, M, act, Y, st);
  if (p.decode) return colpar_decode(s, d, p, X, M, act, Y, reinterpret_cast<float *>(ws_col), st);
  return colpar_tc(s, d, X, M, act_epi(act), Y, s->Fs, st);
}

tp_status_t rowpar_any(const tp_shards *s, const DevState *d, const MlpPlan &p, const void *Y,
                       int64_t M, float *Z, char *ws_row, cudaStream_t st, const Residual &res = Residual()) {
  float *P = reinterpret_cast<float *>(ws_row);
  if (p.simt || p.decode) {
    TP_TRY(p.simt ? rowpar_simt(s, d, p, Y, M, Z, P, st) : rowpar_decode(s, d, p, Y, M, Z, P, st));
    return apply_residual(d, Z, M * s->H, res, st);
  }
  CUtensorMap my;
  TP_TRY(make_map(&my, Y, s->Fs, M, s->T, s->Fs * 2, M * s->Fs * 2, 128));
  return rowpar_tc(s, d, my, 1, M, p.slots2, P, Z, st, res);
}

tp_status_t check_handle(const tp_shards *s, int kind, DevState **d) {
  if (!s || s->kind != kind) return TP_ERR_ARG;
  int dev = 0;
  TP_TRY(dev_state(d, &dev));
  if (dev != s->device) return TP_ERR_ARG;
  return TP_OK;
}

bool valid_variant(tp_variant_t v) {
  return v == TP_VAR_AUTO || v == TP_VAR_PARTIALS || v == TP_VAR_TMEM_ACC;
}

// Workspace: the caller's, or one allocated stream-ordered for this call.
struct Workspace {
  char *ptr = nullptr;
  bool owned = false;
  cudaStream_t st = nullptr;
  ~Workspace() {
    if (owned && ptr) cudaFreeAsync(ptr, st);
  }
};

tp_status_t get_ws(Workspace *w, void *given, size_t given_bytes, size_t need, cudaStream_t st) {
  w->st = st;
  if (given) {
    if (given_bytes < need) return TP_ERR_WORKSPACE;
    if (!aligned16(given)) return TP_ERR_ARG;
    w->ptr = static_cast<char *>(given);
    return TP_OK;
  }
  if (need == 0) return TP_OK;
  void *p = nullptr;
  if (lib_malloc_async(&p, need, st) != cudaSuccess) return TP_ERR_OOM;
  w->ptr = static_cast<char *>(p);
  w->owned = true;
  return TP_OK;
}

// One tensor-core GEMM D[rows x N] over a K axis of nseg segments of kps
// k-tiles: picks CTA-pair or single-CTA tiles and fills the work fields.
struct GemmCall {
  const CUtensorMap *a = nullptr;
  int a_seg = 0;
  const CUtensorMap *b_bn = nullptr, *b_128 = nullptr;  // B maps with box bn rows / 128 rows
  int b_seg = 0;
  int a_mn_seg = 0, b_mn_seg = 0;  // EPI_F32_MN: MN rows per segment of A / B
  int64_t rows = 0, N = 0;
  int bn = 256, kps = 0, nseg = 1, slots = 1;
  Epi epi = EPI_F32;
  BTensor bt{};  // B's tensor (base non-null): EPI_F32 with one slot may take the wide schedule
};

tp_status_t run_gemm(const DevState *d, const GemmCall &c, GemmArgs g, cudaStream_t st) {
  const bool pair = use_pair(c.bn, c.rows);
  g.m_tiles = static_cast<int>(cdiv(c.rows, pair ? 256 : 128));
  g.n_tiles = static_cast<int>(c.N / c.bn);
  g.slots = c.slots;
  g.kt_per_seg = c.kps;
  g.kt_total = c.nseg * c.kps;
  g.kt_per_slot = g.kt_total / c.slots;
  g.a_seg = c.a_seg;
  g.b_seg = c.b_seg;
  g.a_mn_seg = c.a_mn_seg;
  g.b_mn_seg = c.b_mn_seg;
  g.rows_valid = static_cast<int>(c.rows);
  g.cols_valid = static_cast<int>(c.N);
  bool done = false;
  if (pair && c.epi == EPI_F32 && c.slots == 1 && c.bt.base)
    TP_TRY(try_wide(d, c.epi, g, c.N, *c.a, *c.b_128, c.bt, st, &done));
  if (done) return TP_OK;
  if (pair) TP_CUDA(launch_gemm(CFG_PAIR_N256, c.epi, *c.a, *c.b_128, g, d->sms, st));
  else TP_CUDA(launch_gemm(cfg_for(c.bn), c.epi, *c.a, *c.b_bn, g, d->sms, st));
  return TP_OK;
}

int bn_for(int64_t n) { return n % 256 == 0 ? 256 : 128; }

struct TrainPlan {
  int slots2 = 1;       // forward row-parallel slots
  int slots_dx = 1;     // backward dX slots
  int nseg = 1;         // segments of dP (T, or 2T for SwiGLU: dG shards then dU shards)
  size_t fwd_row = 0;   // forward: row-parallel partials
  size_t dP = 0, dx_part = 0;
  size_t fwd_total() const { return round256(fwd_row); }
  size_t bwd_total() const { return round256(dP) + round256(dx_part); }
};

void plan_train(const tp_shards *s, int64_t M, tp_variant_t v, const DevState *d, TrainPlan *p) {
  *p = TrainPlan();
  const int64_t H = s->H, Fs = s->Fs, T = s->T;
  MlpPlan fp;
  plan_mlp(s, M > kDecodeMaxM ? M : kDecodeMaxM + 1, v, d, &fp);
  p->slots2 = fp.slots2;
  p->fwd_row = p->slots2 > 1 ? static_cast<size_t>(p->slots2 * M * H) * 4 : 0;
  p->nseg = static_cast<int>(s->act == TP_ACT_SWIGLU ? 2 * T : T);
  p->slots_dx = (v == TP_VAR_PARTIALS) ? p->nseg : 1;
  p->dP = static_cast<size_t>(p->nseg * M * Fs) * 2;
  p->dx_part = p->slots_dx > 1 ? static_cast<size_t>(p->slots_dx * M * H) * 4 : 0;
}

tp_status_t mlp_forward_train_impl(tp_shards *s, const void *X, int64_t M, tp_act_t act, tp_variant_t v,
                                   float *Z, void *Hsave, void *Psave, void *workspace, size_t ws_bytes,
                                   cudaStream_t st) {
  DevState *d = nullptr;
  TP_TRY(check_handle(s, 0, &d));
  if (s->dt != TP_BF16) return TP_ERR_DTYPE;
  if (M < 0 || !valid_variant(v) || act != s->act) return TP_ERR_ARG;
  if (M == 0) return TP_OK;
  if (!X || !Z || !Hsave || !aligned16(X) || !aligned16(Z) || !aligned16(Hsave)) return TP_ERR_ARG;
  if (act != TP_ACT_IDENTITY && (!Psave || !aligned16(Psave))) return TP_ERR_ARG;
  if (M > (1LL << 30)) return TP_ERR_UNSUPPORTED;
  TrainPlan p;
  plan_train(s, M, v, d, &p);
  Workspace w;
  TP_TRY(get_ws(&w, workspace, ws_bytes, p.fwd_total(), st));
  const int64_t H = s->H, T = s->T, Fs = s->Fs;
  CUtensorMap mx;
  TP_TRY(make_map(&mx, X, H, M, 1, H * 2, M * H * 2, 128));
  GemmArgs g = base_args(d);
  g.out = Hsave;
  g.ld_out = Fs;
  g.shard_stride = M * Fs;
  g.shard_cols = static_cast<int>(Fs);
  GemmCall c;
  c.a = &mx;
  c.b_bn = &s->map_w1_b;
  c.b_128 = &s->map_w1_a;
  c.b_seg = kKtileBlocked;
  c.rows = M;
  c.N = T * s->R1;
  c.bn = s->bn1;
  c.kps = static_cast<int>(H / 64);
  if (act == TP_ACT_GELU_ERF) {
    c.epi = EPI_GELU_SAVE_BF16;
    g.out2 = Psave;
  } else if (act == TP_ACT_SWIGLU) {
    c.epi = EPI_SWIGLU_SAVE_BF16;
    g.out2 = Psave;
    g.out3 = static_cast<char *>(Psave) + static_cast<size_t>(T * M * Fs) * 2;
  } else {
    c.epi = EPI_IDENT_BF16;
  }
  TP_TRY(run_gemm(d, c, g, st));
  CUtensorMap mh;
  TP_TRY(make_map(&mh, Hsave, Fs, M, T, Fs * 2, M * Fs * 2, 128));
  return rowpar_tc(s, d, mh, 1, M, p.slots2, reinterpret_cast<float *>(w.ptr), Z, st);
}

tp_status_t mlp_backward_impl(tp_shards *s, const void *X, const void *Hsave, const void *Psave,
                              const void *dZ, int64_t M, tp_variant_t v, float *dX, float *dW1, float *dW2,
                              void *workspace, size_t ws_bytes, cudaStream_t st) {
  DevState *d = nullptr;
  TP_TRY(check_handle(s, 0, &d));
  if (!s->backward) return TP_ERR_ARG;
  if (M < 0 || !valid_variant(v)) return TP_ERR_ARG;
  if (M == 0) return TP_OK;
  for (const void *ptr : {X, Hsave, dZ, static_cast<const void *>(dX), static_cast<const void *>(dW1),
                          static_cast<const void *>(dW2)})
    if (!ptr || !aligned16(ptr)) return TP_ERR_ARG;
  if (s->act != TP_ACT_IDENTITY && (!Psave || !aligned16(Psave))) return TP_ERR_ARG;
  if (M > (1LL << 30)) return TP_ERR_UNSUPPORTED;
  TrainPlan p;
  plan_train(s, M, v, d, &p);
  Workspace w;
  TP_TRY(get_ws(&w, workspace, ws_bytes, p.bwd_total(), st));
  const int64_t H = s->H, T = s->T, Fs = s->Fs, F = s->F;
  const int64_t ncols = p.nseg * Fs;
  char *dP = w.ptr;
  float *dxp = reinterpret_cast<float *>(dP + round256(p.dP));

  // 1. dH = dZ W2^T for every shard, times the activation's derivative -> dP
  CUtensorMap mdz;
  TP_TRY(make_map(&mdz, dZ, H, M, 1, H * 2, M * H * 2, 128));
  {
    GemmArgs g = base_args(d);
    g.out = dP;
    g.ld_out = Fs;
    g.shard_stride = M * Fs;
    g.shard_cols = static_cast<int>(Fs);
    GemmCall c;
    c.a = &mdz;
    c.b_bn = &s->map_w2o_bn;
    c.b_128 = &s->map_w2o_128;
    c.rows = M;
    c.N = F;
    c.bn = s->bn_dh;
    c.kps = static_cast<int>(H / 64);
    if (s->act == TP_ACT_GELU_ERF) {
      c.epi = EPI_DGELU_BF16;
      g.aux = Psave;
    } else if (s->act == TP_ACT_SWIGLU) {
      c.epi = EPI_DSWIGLU_BF16;
      g.out2 = dP + static_cast<size_t>(T * M * Fs) * 2;
      g.aux = Psave;
      g.aux2 = static_cast<const char *>(Psave) + static_cast<size_t>(T * M * Fs) * 2;
    } else {
      c.epi = EPI_IDENT_BF16;
    }
    TP_TRY(run_gemm(d, c, g, st));
  }
  // 2. dX = sum over shards of dP_i W1_i^T (the backward all-reduce-sum)
  CUtensorMap mdp;
  TP_TRY(make_map(&mdp, dP, Fs, M, p.nseg, Fs * 2, M * Fs * 2, 128));
  {
    GemmArgs g = base_args(d);
    g.out = p.slots_dx > 1 ? static_cast<void *>(dxp) : static_cast<void *>(dX);
    g.ld_out = H;
    g.slot_stride = M * H;
    GemmCall c;
    c.a = &mdp;
    c.a_seg = 1;
    c.b_bn = &s->map_w1o_bn;
    c.b_128 = &s->map_w1o_128;
    c.bt = BTensor{s->w1o, static_cast<uint64_t>(ncols), static_cast<uint64_t>(H), 1, static_cast<uint64_t>(ncols) * 2,
                   static_cast<uint64_t>(H * ncols) * 2};
    c.rows = M;
    c.N = H;
    c.bn = s->bn2;
    c.kps = static_cast<int>(Fs / 64);
    c.nseg = p.nseg;
    c.slots = p.slots_dx;
    TP_TRY(run_gemm(d, c, g, st));
    if (p.slots_dx > 1) TP_CUDA(launch_shard_sum_strided(dxp, p.slots_dx, M * H, M * H, dX, d->sms, st));
  }
  // 3. dW2 = H^T dZ  [F x H];  4. dW1 = X^T dP  [H x ncols].  K is the token axis, so every
  // operand is read MN-major straight from its [tokens][features] layout (64 x 64 boxes; the
  // copies fill tokens past M with zeros): per-shard H and dP as [segments][M][Fs].
  // Each copy fetches two 64-row MN blocks (4-D maps, kMnPairBox): half the copy instructions
  // per stage, which is what bounds these GEMMs' loads.  Both blocks lie in one segment, since
  // shard widths and H are multiples of 128 (tp_shard_weights requires it for bf16).
  if (Fs % 128 != 0 || H % 128 != 0) return TP_ERR_UNSUPPORTED;
  CUtensorMap m_h, m_x, m_dz, m_dp;
  TP_TRY(make_map_mn_pairs(&m_h, Hsave, Fs, M, T));
  TP_TRY(make_map_mn_pairs(&m_x, X, H, M, 1));
  TP_TRY(make_map_mn_pairs(&m_dz, dZ, H, M, 1));
  TP_TRY(make_map_mn_pairs(&m_dp, dP, Fs, M, p.nseg));
  const int ktok = static_cast<int>(cdiv(M, 64));
  {
    GemmArgs g = base_args(d);
    g.out = dW2;
    g.ld_out = H;
    GemmCall c;
    c.a = &m_h;
    c.a_mn_seg = static_cast<int>(Fs);
    c.b_bn = c.b_128 = &m_dz;
    c.rows = F;
    c.N = H;
    c.bn = bn_for(H);
    c.kps = ktok;
    c.epi = EPI_F32_MN;
    TP_TRY(run_gemm(d, c, g, st));
  }
  {
    GemmArgs g = base_args(d);
    g.out = dW1;
    g.ld_out = ncols;
    GemmCall c;
    c.a = &m_x;
    c.b_bn = c.b_128 = &m_dp;
    c.b_mn_seg = static_cast<int>(Fs);
    c.rows = H;
    c.N = ncols;
    c.bn = bn_for(ncols);
    c.kps = ktok;
    c.epi = EPI_F32_MN;
    TP_TRY(run_gemm(d, c, g, st));
  }
  return TP_OK;
}

bool act_ok(const tp_shards *s, tp_act_t act) {
  if (act == s->act) return true;
  return s->act != TP_ACT_SWIGLU && (act == TP_ACT_GELU_ERF || act == TP_ACT_IDENTITY);
}

tp_status_t mlp_forward_impl(tp_shards *s, const void *X, int64_t M, tp_act_t act, tp_variant_t v,
                             float *Z, void *workspace, size_t ws_bytes, cudaStream_t st,
                             const Residual &res = Residual(), size_t budget = 0) {
  DevState *d = nullptr;
  TP_TRY(check_handle(s, 0, &d));
  if (M < 0 || !valid_variant(v) || !act_ok(s, act)) return TP_ERR_ARG;
  if (M == 0) return TP_OK;
  if (!X || !Z || !aligned16(X) || !aligned16(Z)) return TP_ERR_ARG;
  if (M > (1LL << 30)) return TP_ERR_UNSUPPORTED;
  MlpPlan p;
  TP_TRY(plan_mlp(s, M, v, d, &p, budget));
  Workspace w;
  TP_TRY(get_ws(&w, workspace, ws_bytes, p.total(), st));
  char *Y = w.ptr;
  char *ws_col = Y + round256(p.y_bytes);
  char *ws_row = ws_col + round256(p.col_bytes);
  TP_TRY(colpar_any(s, d, p, X, M, act, Y, ws_col, st));
  return rowpar_any(s, d, p, Y, M, Z, ws_row, st, res);
}

// ---- one tensor-parallel transformer block ---------------------------------------

// Attention core (the block's, and tp_attention_forward): the fused kernel
// reads head-major Q, K and V [heads][M][128] through TMA (V in 64 x 64 boxes,
// as the P V product's MN-major operand).  The maps' key extent is M, so the
// copy engine fills keys past M with zeros.
tp_status_t attention_core(const DevState *d, const void *Q, const void *K, const void *V, int64_t M,
                           int64_t heads, int causal, void *O, int64_t ldo, cudaStream_t st) {
  const int64_t hd = kAttnHeadDim;
  CUtensorMap mq, mk, mv;
  TP_TRY(make_map(&mq, Q, hd, M, heads, hd * 2, M * hd * 2, 128));
  TP_TRY(make_map(&mk, K, hd, M, heads, hd * 2, M * hd * 2, static_cast<uint32_t>(attention_key_box_rows())));
  TP_TRY(make_map(&mv, V, hd, M, heads, hd * 2, M * hd * 2, 64));
  AttnArgs g;
  std::memset(&g, 0, sizeof g);
  g.M = static_cast<int>(M);
  g.heads = static_cast<int>(heads);
  g.m_tiles = static_cast<int>(cdiv(M, 128));
  g.causal = causal ? 1 : 0;
  g.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(hd));
  g.O = O;
  g.ldo = ldo;
  g.status = d->status;
  g.wait_limit_ns = g_wait_ns.load();
  TP_CUDA(launch_attention(mq, mk, mv, g, d->sms, st));
  return TP_OK;
}

struct BlockPlan {
  int slots_o = 1;  // O-projection accumulation slots
  MlpPlan mlp;
  size_t qkv = 0, O = 0, opart = 0, h = 0, hb = 0;
  size_t total() const {
    return round256(qkv) + round256(O) + round256(opart) + round256(h) + round256(hb) + mlp.total();
  }
};

void plan_block(const tp_shards *a, const tp_shards *m, int64_t M, tp_variant_t v, const DevState *d, BlockPlan *p) {
  *p = BlockPlan();
  const int64_t H = a->H;
  p->slots_o = v == TP_VAR_PARTIALS ? a->T : 1;
  plan_mlp(m, M, v, d, &p->mlp);
  p->qkv = static_cast<size_t>(3 * H * M) * 2;  // Q, K and V head-major
  p->O = static_cast<size_t>(M * H) * 2;
  p->opart = p->slots_o > 1 ? static_cast<size_t>(p->slots_o * M * H) * 4 : 0;
  p->h = static_cast<size_t>(M * H) * 4;
  p->hb = static_cast<size_t>(M * H) * 2;
}

tp_status_t block_forward_impl(tp_shards *a, tp_shards *m, const void *X, int64_t M, int causal,
                               tp_variant_t v, float *out, float *h_out, void *workspace, size_t ws_bytes,
                               cudaStream_t st) {
  DevState *d = nullptr;
  TP_TRY(check_handle(a, 1, &d));
  TP_TRY(check_handle(m, 0, &d));
  if (m->dt != TP_BF16) return TP_ERR_DTYPE;
  if (m->H != a->H || m->T != a->T || M < 0 || !valid_variant(v)) return TP_ERR_ARG;
  if (a->head_dim != kAttnHeadDim) return TP_ERR_UNSUPPORTED;
  if (M == 0) return TP_OK;
  if (!X || !out || !aligned16(X) || !aligned16(out) || (h_out && !aligned16(h_out))) return TP_ERR_ARG;
  if (M > (1LL << 24)) return TP_ERR_UNSUPPORTED;
  BlockPlan p;
  plan_block(a, m, M, v, d, &p);
  Workspace w;
  TP_TRY(get_ws(&w, workspace, ws_bytes, p.total(), st));
  const int64_t H = a->H, nh = a->n_heads, hd = a->head_dim;
  char *qkv = w.ptr;
  char *O = qkv + round256(p.qkv);
  float *opart = reinterpret_cast<float *>(O + round256(p.O));
  float *h = reinterpret_cast<float *>(reinterpret_cast<char *>(opart) + round256(p.opart));
  char *hb = reinterpret_cast<char *>(h) + round256(p.h);
  char *mws = hb + round256(p.hb);
  if (h_out) h = h_out;

  // 1. QKV projection of every shard: Q, K and V head-major [3][nh][M][hd]
  CUtensorMap mx;
  TP_TRY(make_map(&mx, X, H, M, 1, H * 2, M * H * 2, 128));
  {
    GemmArgs g = base_args(d);
    g.out = qkv;
    g.shard_cols = static_cast<int>(a->R1);
    g.head_dim = static_cast<int>(hd);
    g.n_heads = static_cast<int>(nh);
    GemmCall c;
    c.a = &mx;
    c.b_bn = &a->map_w1_b;
    c.b_128 = &a->map_w1_a;
    c.b_seg = kKtileBlocked;
    c.rows = M;
    c.N = a->T * a->R1;
    c.bn = a->bn1;
    c.kps = static_cast<int>(H / 64);
    c.epi = EPI_QKV_HEADS_BF16;
    TP_TRY(run_gemm(d, c, g, st));
  }
  const size_t head_block = static_cast<size_t>(nh * M * hd) * 2;
  const char *Q = qkv, *K = qkv + head_block, *V = qkv + 2 * head_block;
  // 2.-5. causal attention per head, fused: O [M x H], heads side by side
  TP_TRY(attention_core(d, Q, K, V, M, nh, causal, O, H, st));
  // 6. row-parallel output projection + all-reduce-sum #1, 7. residual: h = X + the sum,
  //    hb = bf16(h) (fused into the GEMM's epilogue when it accumulates all shards in TMEM)
  CUtensorMap mo;
  TP_TRY(make_map(&mo, O, H, M, 1, H * 2, M * H * 2, 128));
  Residual r1;
  r1.add_bf16 = X;
  r1.out_bf16 = hb;
  TP_TRY(rowpar_tc(a, d, mo, 0, M, p.slots_o, opart, h, st, r1));
  // 8. the MLP on the residual stream + all-reduce-sum #2, 9. residual: out = h + the sum
  Residual r2;
  r2.add_f32 = h;
  TP_TRY(mlp_forward_impl(m, hb, M, m->act, v, out, mws, p.mlp.total(), st, r2));
  return TP_OK;
}

}  // namespace

bool tp::encode_store_map(CUtensorMap *m, const void *base, int elem_bytes, uint64_t d0, uint64_t d1, uint64_t d2,
                          uint64_t s1, uint64_t s2, uint32_t box0, uint32_t box1) {
  EncodeTiledFn f = encode_fn();
  if (!f || (elem_bytes != 2 && elem_bytes != 4)) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return f(m, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
           const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t tp::mlp_workspace_within(tp_shards *s, int64_t M, size_t budget) {
  DevState *d = nullptr;
  if (!s || s->kind != 0 || M <= 0 || budget == 0 || dev_state(&d) != TP_OK) return 0;
  MlpPlan p;
  if (plan_mlp(s, M, TP_VAR_AUTO, d, &p, budget) != TP_OK) return 0;
  return p.total();
}

tp_status_t tp::mlp_forward_within(tp_shards *s, const void *X, int64_t M, tp_act_t act, float *Z, void *ws,
                                   size_t budget, cudaStream_t st) {
  if (budget == 0) return TP_ERR_ARG;
  return mlp_forward_impl(s, X, M, act, TP_VAR_AUTO, Z, ws, budget, st, Residual(), budget);
}

bool tp::handle_ready_on_current_device(const tp_shards *s) {
  int dev = 0;
  if (!s || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  if (dev != s->device) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  return g_dev[dev].ready;
}

// ============================================================================
// C ABI
// ============================================================================

extern "C" {

const char *tp_status_str(tp_status_t s) {
  switch (s) {
    case TP_OK: return "TP_OK";
    case TP_ERR_ARG: return "TP_ERR_ARG: invalid argument";
    case TP_ERR_INDIVISIBLE: return "TP_ERR_INDIVISIBLE: dimension not divisible by the shard count";
    case TP_ERR_DTYPE: return "TP_ERR_DTYPE: element type not supported";
    case TP_ERR_ARCH: return "TP_ERR_ARCH: current device is not sm_103 (GB300)";
    case TP_ERR_OOM: return "TP_ERR_OOM: allocation failed";
    case TP_ERR_CUDA: return "TP_ERR_CUDA: CUDA call failed";
    case TP_ERR_TIMEOUT: return "TP_ERR_TIMEOUT: a device-side wait ran out";
    case TP_ERR_DEVICE_CHECK: return "TP_ERR_DEVICE_CHECK: a device-side check failed";
    case TP_ERR_UNSUPPORTED: return "TP_ERR_UNSUPPORTED: shape not supported by the kernels";
    case TP_ERR_WORKSPACE: return "TP_ERR_WORKSPACE: workspace too small";
  }
  return "unknown tp_status_t";
}

int tp_abi_version(void) { return TP_ABI_VERSION; }

tp_status_t tp_inject_alloc_failures(int count) {
  if (count < 0) return TP_ERR_ARG;
  g_fail_allocs.store(count);
  return TP_OK;
}

tp_status_t tp_set_machine_balance(double flop_per_byte) {
  if (!(flop_per_byte >= 0.0) || flop_per_byte > 1e6) return TP_ERR_ARG;
  g_balance_override.store(flop_per_byte);
  return TP_OK;
}

tp_status_t tp_set_rowpar_schedule(int wide) {
  if (wide != 0 && wide != 1) return TP_ERR_ARG;
  g_rowpar_wide.store(wide);
  return TP_OK;
}

tp_status_t tp_set_wait_limit_ns(uint64_t ns) {
  g_wait_ns.store(ns == 0 ? kDefaultWaitNs : ns);
  return TP_OK;
}

tp_status_t tp_shard_weights(const void *W1, const void *W2, int64_t H, int64_t F, int T,
                             tp_act_t act, tp_dtype_t dt, void *stream, tp_shards_t *out) {
  if (!out) return TP_ERR_ARG;
  *out = nullptr;
  if (!W1 || !W2 || H <= 0 || F <= 0 || T < 1 || T > kMaxShards) return TP_ERR_ARG;
  if (act != TP_ACT_GELU_ERF && act != TP_ACT_SWIGLU && act != TP_ACT_IDENTITY) return TP_ERR_ARG;
  if (dt != TP_F32 && dt != TP_BF16) return TP_ERR_DTYPE;
  if (F % T != 0) return TP_ERR_INDIVISIBLE;
  const int64_t Fs = F / T;
  const size_t eb = esize(dt);
  if ((reinterpret_cast<uintptr_t>(W1) | reinterpret_cast<uintptr_t>(W2)) % eb) return TP_ERR_ARG;
  if (dt == TP_BF16 && (H % 128 != 0 || Fs % 128 != 0)) return TP_ERR_UNSUPPORTED;
  if (act == TP_ACT_SWIGLU && Fs % kSwigluGranule != 0) return TP_ERR_UNSUPPORTED;
  if (H > (1LL << 31) || F > (1LL << 31)) return TP_ERR_UNSUPPORTED;
  DevState *d = nullptr;
  int dev = 0;
  TP_TRY(dev_state(&d, &dev));
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  tp_shards *s = new (std::nothrow) tp_shards();
  if (!s) return TP_ERR_OOM;
  s->kind = 0;
  s->device = dev;
  s->H = H;
  s->F = F;
  s->Fs = Fs;
  s->T = T;
  s->act = act;
  s->dt = dt;
  s->R1 = act == TP_ACT_SWIGLU ? 2 * Fs : Fs;
  const size_t b1 = static_cast<size_t>(T * s->R1 * H) * eb, b2 = static_cast<size_t>(T * H * Fs) * eb;
  if (lib_malloc(&s->w1p, b1) != cudaSuccess || lib_malloc(&s->w2p, b2) != cudaSuccess) {
    tp_shards_destroy(s);
    return TP_ERR_OOM;
  }
  tp_status_t r = cuda_status(launch_pack(act == TP_ACT_SWIGLU ? PACK_W1_SWIGLU : PACK_W1, W1,
                                          act == TP_ACT_SWIGLU ? 2 * F : F, s->w1p, T, s->R1, H,
                                          static_cast<int>(eb), F, 0, Fs, st));
  if (r == TP_OK)
    r = cuda_status(launch_pack(PACK_ROWS, W2, H, s->w2p, T, H, Fs, static_cast<int>(eb), 0, 0, 0, st));
  if (r == TP_OK && dt == TP_BF16) {
    s->bn1 = (act == TP_ACT_SWIGLU || Fs % 256 == 0) ? 256 : 128;
    s->bn2 = (H % 256 == 0) ? 256 : 128;
    r = make_weight_maps(s, Fs);
  }
  if (r != TP_OK) {
    tp_shards_destroy(s);
    return r;
  }
  *out = s;
  return TP_OK;
}

tp_status_t tp_shard_weights_qkv(const void *Wqkv, const void *Wo, int64_t H, int n_heads,
                                 int head_dim, int T, void *stream, tp_shards_t *out) {
  if (!out) return TP_ERR_ARG;
  *out = nullptr;
  if (!Wqkv || !Wo || H <= 0 || n_heads <= 0 || head_dim <= 0 || T < 1 || T > kMaxShards)
    return TP_ERR_ARG;
  if (static_cast<int64_t>(n_heads) * head_dim != H) return TP_ERR_ARG;
  if (n_heads % T != 0) return TP_ERR_INDIVISIBLE;
  const int64_t W = static_cast<int64_t>(n_heads / T) * head_dim;
  if ((reinterpret_cast<uintptr_t>(Wqkv) | reinterpret_cast<uintptr_t>(Wo)) % 2) return TP_ERR_ARG;
  if (H % 128 != 0 || W % 64 != 0 || (3 * W) % 128 != 0) return TP_ERR_UNSUPPORTED;
  DevState *d = nullptr;
  int dev = 0;
  TP_TRY(dev_state(&d, &dev));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  tp_shards *s = new (std::nothrow) tp_shards();
  if (!s) return TP_ERR_OOM;
  s->kind = 1;
  s->device = dev;
  s->H = H;
  s->F = H;
  s->Fs = W;
  s->T = T;
  s->act = TP_ACT_IDENTITY;
  s->dt = TP_BF16;
  s->n_heads = n_heads;
  s->head_dim = head_dim;
  s->R1 = 3 * W;
  const size_t b1 = static_cast<size_t>(T * s->R1 * H) * 2, b2 = static_cast<size_t>(T * H * W) * 2;
  if (lib_malloc(&s->w1p, b1) != cudaSuccess || lib_malloc(&s->w2p, b2) != cudaSuccess) {
    tp_shards_destroy(s);
    return TP_ERR_OOM;
  }
  tp_status_t r = cuda_status(launch_pack(PACK_QKV, Wqkv, 3 * H, s->w1p, T, s->R1, H, 2, 0, H, W, st));
  if (r == TP_OK) r = cuda_status(launch_pack(PACK_ROWS, Wo, H, s->w2p, T, H, W, 2, 0, 0, 0, st));
  if (r == TP_OK) {
    s->bn1 = ((3 * W) % 256 == 0) ? 256 : 128;
    s->bn2 = (H % 256 == 0) ? 256 : 128;
    r = make_weight_maps(s, W);
  }
  if (r != TP_OK) {
    tp_shards_destroy(s);
    return r;
  }
  *out = s;
  return TP_OK;
}

tp_status_t tp_shard_get(tp_shards_t s, int i, int which, void *host_dst) {
  if (!s || !host_dst || i < 0 || i >= s->T) return TP_ERR_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TP_ERR_CUDA;
  if (dev != s->device) return TP_ERR_ARG;
  const size_t eb = esize(s->dt);
  PackMode mode;
  const void *packed;
  int64_t R, K, W, elems;
  int wh = 0;
  if (which == 2) {
    mode = PACK_ROWS;
    packed = s->w2p;
    R = s->H;
    K = s->Fs;
    W = 0;
    elems = s->Fs * s->H;
  } else if (which == 0 || which == 1) {
    if (s->kind == 1) {
      if (which != 0) return TP_ERR_ARG;
      mode = PACK_QKV;
      elems = s->H * 3 * s->Fs;
    } else {
      if (which == 1 && s->act != TP_ACT_SWIGLU) return TP_ERR_ARG;
      mode = s->act == TP_ACT_SWIGLU ? PACK_W1_SWIGLU : PACK_W1;
      elems = s->H * s->Fs;
      wh = which;
    }
    packed = s->w1p;
    R = s->R1;
    K = s->H;
    W = s->Fs;
  } else {
    return TP_ERR_ARG;
  }
  void *tmp = nullptr;
  if (lib_malloc(&tmp, static_cast<size_t>(elems) * eb) != cudaSuccess) return TP_ERR_OOM;
  tp_status_t r = cuda_status(launch_unpack(mode, packed, tmp, i, s->T, wh, R, K, static_cast<int>(eb), W, 0));
  if (r == TP_OK) r = cuda_status(cudaMemcpy(host_dst, tmp, static_cast<size_t>(elems) * eb,
                                             cudaMemcpyDeviceToHost));
  cudaFree(tmp);
  return r;
}

tp_status_t tp_shard_info(tp_shards_t s, int *kind, int64_t *H, int64_t *F, int *T, int *act,
                          int *dtype) {
  if (!s) return TP_ERR_ARG;
  if (kind) *kind = s->kind;
  if (H) *H = s->H;
  if (F) *F = s->F;
  if (T) *T = s->T;
  if (act) *act = s->act;
  if (dtype) *dtype = s->dt;
  return TP_OK;
}

void tp_shards_destroy(tp_shards_t s) {
  if (!s) return;
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != s->device) cudaSetDevice(s->device);
  cudaDeviceSynchronize();
  if (s->w1p) cudaFree(s->w1p);
  if (s->w2p) cudaFree(s->w2p);
  if (s->w1o) cudaFree(s->w1o);
  if (s->w2o) cudaFree(s->w2o);
  if (prev >= 0 && prev != s->device) cudaSetDevice(prev);
  delete s;
}

tp_status_t tp_shards_enable_backward(tp_shards_t s, const void *W1, const void *W2, void *stream) {
  if (!s || s->kind != 0 || !W1 || !W2) return TP_ERR_ARG;
  if (s->dt != TP_BF16) return TP_ERR_DTYPE;
  if (!aligned16(W1) || !aligned16(W2)) return TP_ERR_ARG;
  DevState *d = nullptr;
  TP_TRY(check_handle(s, 0, &d));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t H = s->H, F = s->F, ncols = s->act == TP_ACT_SWIGLU ? 2 * F : F;
  const size_t b1 = static_cast<size_t>(H * ncols) * 2, b2 = static_cast<size_t>(F * H) * 2;
  if (!s->w1o && lib_malloc(&s->w1o, b1) != cudaSuccess) return TP_ERR_OOM;
  if (!s->w2o && lib_malloc(&s->w2o, b2) != cudaSuccess) return TP_ERR_OOM;
  TP_CUDA(cudaMemcpyAsync(s->w1o, W1, b1, cudaMemcpyDeviceToDevice, st));
  TP_CUDA(cudaMemcpyAsync(s->w2o, W2, b2, cudaMemcpyDeviceToDevice, st));
  s->bn_dh = s->Fs % 256 == 0 ? 256 : 128;
  TP_TRY(make_map(&s->map_w2o_bn, s->w2o, H, F, 1, H * 2, F * H * 2, s->bn_dh));
  TP_TRY(make_map(&s->map_w2o_128, s->w2o, H, F, 1, H * 2, F * H * 2, 128));
  TP_TRY(make_map(&s->map_w1o_bn, s->w1o, ncols, H, 1, ncols * 2, H * ncols * 2, s->bn2));
  TP_TRY(make_map(&s->map_w1o_128, s->w1o, ncols, H, 1, ncols * 2, H * ncols * 2, 128));
  s->backward = true;
  return TP_OK;
}

size_t tp_mlp_train_workspace_bytes(tp_shards_t s, int64_t M, tp_variant_t v) {
  DevState *d = nullptr;
  if (!s || s->kind != 0 || M <= 0 || !valid_variant(v) || dev_state(&d) != TP_OK) return 0;
  TrainPlan p;
  plan_train(s, M, v, d, &p);
  return p.fwd_total();
}

tp_status_t tp_mlp_forward_train(tp_shards_t s, const void *X, int64_t M, tp_act_t act, tp_variant_t v,
                                 float *Z, void *Hsave, void *Psave, void *workspace, size_t ws_bytes,
                                 void *stream) {
  return mlp_forward_train_impl(s, X, M, act, v, Z, Hsave, Psave, workspace, ws_bytes,
                                static_cast<cudaStream_t>(stream));
}

size_t tp_mlp_backward_workspace_bytes(tp_shards_t s, int64_t M, tp_variant_t v) {
  DevState *d = nullptr;
  if (!s || s->kind != 0 || M <= 0 || !valid_variant(v) || dev_state(&d) != TP_OK) return 0;
  TrainPlan p;
  plan_train(s, M, v, d, &p);
  return p.bwd_total();
}

tp_status_t tp_mlp_backward(tp_shards_t s, const void *X, const void *Hsave, const void *Psave,
                            const void *dZ, int64_t M, tp_variant_t v, float *dX, float *dW1, float *dW2,
                            void *workspace, size_t ws_bytes, void *stream) {
  return mlp_backward_impl(s, X, Hsave, Psave, dZ, M, v, dX, dW1, dW2, workspace, ws_bytes,
                           static_cast<cudaStream_t>(stream));
}

size_t tp_mlp_workspace_bytes(tp_shards_t s, int64_t M, tp_variant_t v) {
  DevState *d = nullptr;
  if (!s || s->kind != 0 || M <= 0 || !valid_variant(v) || dev_state(&d) != TP_OK) return 0;
  MlpPlan p;
  if (plan_mlp(s, M, v, d, &p) != TP_OK) return 0;
  return p.total();
}

size_t tp_colpar_workspace_bytes(tp_shards_t s, int64_t M) {
  DevState *d = nullptr;
  if (!s || s->kind != 0 || M <= 0 || dev_state(&d) != TP_OK) return 0;
  MlpPlan p;
  if (plan_mlp(s, M, TP_VAR_AUTO, d, &p) != TP_OK) return 0;
  return p.col_bytes;
}

tp_status_t tp_colpar_forward(tp_shards_t s, const void *X, int64_t M, tp_act_t act, void *Y,
                              void *workspace, size_t ws_bytes, void *stream) {
  DevState *d = nullptr;
  TP_TRY(check_handle(s, 0, &d));
  if (M < 0 || !act_ok(s, act)) return TP_ERR_ARG;
  if (M == 0) return TP_OK;
  if (!X || !Y || !aligned16(X) || !aligned16(Y)) return TP_ERR_ARG;
  if (M > (1LL << 30)) return TP_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MlpPlan p;
  TP_TRY(plan_mlp(s, M, TP_VAR_AUTO, d, &p));
  Workspace w;
  TP_TRY(get_ws(&w, workspace, ws_bytes, p.col_bytes, st));
  return colpar_any(s, d, p, X, M, act, Y, w.ptr, st);
}

size_t tp_rowpar_workspace_bytes(tp_shards_t s, int64_t M, tp_variant_t v) {
  DevState *d = nullptr;
  if (!s || s->kind != 0 || M <= 0 || !valid_variant(v) || dev_state(&d) != TP_OK) return 0;
  MlpPlan p;
  if (plan_mlp(s, M, v, d, &p) != TP_OK) return 0;
  return p.row_bytes;
}

tp_status_t tp_rowpar_tiles(tp_shards_t s, int64_t M, tp_variant_t v, int32_t *out) {
  if (!out) return TP_ERR_ARG;
  out[0] = out[1] = out[2] = 0;
  DevState *d = nullptr;
  TP_TRY(check_handle(s, 0, &d));
  if (M <= 0 || !valid_variant(v)) return TP_ERR_ARG;
  MlpPlan p;
  TP_TRY(plan_mlp(s, M, v, d, &p));
  // the path rowpar_tc takes: tensor cores, CTA pairs, one accumulation slot, float32 output
  if (p.simt || p.decode || p.slots2 != 1 || !use_pair(s->bn2, M) || g_rowpar_wide.load() == 0) return TP_OK;
  const WidePlan wp = plan_wide(static_cast<int>(cdiv(M, 256)), s->H, d->sms / 2, s->T * (s->Fs / 64));
  out[0] = wp.bn;
  out[1] = wp.nb;
  out[2] = wp.q;
  return TP_OK;
}

tp_status_t tp_rowpar_forward(tp_shards_t s, const void *Y, int64_t M, tp_variant_t v, float *Z,
                              void *workspace, size_t ws_bytes, void *stream) {
  DevState *d = nullptr;
  TP_TRY(check_handle(s, 0, &d));
  if (M < 0 || !valid_variant(v)) return TP_ERR_ARG;
  if (M == 0) return TP_OK;
  if (!Y || !Z || !aligned16(Y) || !aligned16(Z)) return TP_ERR_ARG;
  if (M > (1LL << 30)) return TP_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MlpPlan p;
  TP_TRY(plan_mlp(s, M, v, d, &p));
  Workspace w;
  TP_TRY(get_ws(&w, workspace, ws_bytes, p.row_bytes, st));
  return rowpar_any(s, d, p, Y, M, Z, w.ptr, st);
}

tp_status_t tp_mlp_forward(tp_shards_t s, const void *X, int64_t M, tp_act_t act, tp_variant_t v,
                           float *Z, void *workspace, size_t ws_bytes, void *stream) {
  return mlp_forward_impl(s, X, M, act, v, Z, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

size_t tp_mlp_host_workspace_bytes(tp_shards_t s, int64_t M, tp_variant_t v) {
  if (!s || s->kind != 0 || M <= 0) return 0;
  const size_t inner = tp_mlp_workspace_bytes(s, M, v);
  if (inner == 0) return 0;
  return round256(static_cast<size_t>(M * s->H) * esize(s->dt)) + round256(static_cast<size_t>(M * s->H) * 4) +
         inner;
}

tp_status_t tp_mlp_forward_host(tp_shards_t s, const void *X_host, int64_t M, tp_act_t act,
                                tp_variant_t v, float *Z_host, void *workspace, size_t ws_bytes,
                                void *stream) {
  if (!s || s->kind != 0 || M < 0) return TP_ERR_ARG;
  if (M == 0) return TP_OK;
  if (!X_host || !Z_host) return TP_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t need = tp_mlp_host_workspace_bytes(s, M, v);
  if (need == 0) return TP_ERR_ARG;
  Workspace w;
  TP_TRY(get_ws(&w, workspace, ws_bytes, need, st));
  const size_t xb = static_cast<size_t>(M * s->H) * esize(s->dt), zb = static_cast<size_t>(M * s->H) * 4;
  char *Xd = w.ptr;
  float *Zd = reinterpret_cast<float *>(w.ptr + round256(xb));
  char *inner = w.ptr + round256(xb) + round256(zb);
  TP_CUDA(cudaMemcpyAsync(Xd, X_host, xb, cudaMemcpyHostToDevice, st));
  TP_TRY(mlp_forward_impl(s, Xd, M, act, v, Zd, inner, need - round256(xb) - round256(zb), st));
  TP_CUDA(cudaMemcpyAsync(Z_host, Zd, zb, cudaMemcpyDeviceToHost, st));
  return TP_OK;
}

size_t tp_attn_proj_workspace_bytes(tp_shards_t s, int64_t M, tp_variant_t v) {
  DevState *d = nullptr;
  if (!s || s->kind != 1 || M <= 0 || !valid_variant(v) || dev_state(&d) != TP_OK) return 0;
  int slots = 1;
  if (v == TP_VAR_PARTIALS) slots = s->T;
  if (v == TP_VAR_AUTO) {
    slots = choose_slots(cdiv(M, 128) * (s->H / s->bn2), s->T, static_cast<int>(s->Fs / 64), d->sms,
                         ktile_per_partial_byte(d, s->bn2), M * s->H * 4, false);
  }
  return slots > 1 ? round256(static_cast<size_t>(slots * M * s->H) * 4) : 0;
}

tp_status_t tp_attn_proj_forward(tp_shards_t s, const void *X, const void *A, int64_t M,
                                 tp_variant_t v, void *QKV, float *Z, void *workspace,
                                 size_t ws_bytes, void *stream) {
  DevState *d = nullptr;
  TP_TRY(check_handle(s, 1, &d));
  if (M < 0 || !valid_variant(v)) return TP_ERR_ARG;
  if (M == 0) return TP_OK;
  if ((QKV && !X) || (Z && !A) || (!QKV && !Z)) return TP_ERR_ARG;
  if ((X && !aligned16(X)) || (A && !aligned16(A)) || (QKV && !aligned16(QKV)) || (Z && !aligned16(Z)))
    return TP_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (QKV) TP_TRY(colpar_tc(s, d, X, M, EPI_IDENT_BF16, QKV, s->R1, st));
  if (Z) {
    int slots = 1;
    if (v == TP_VAR_PARTIALS) slots = s->T;
    if (v == TP_VAR_AUTO) {
      slots = choose_slots(cdiv(M, 128) * (s->H / s->bn2), s->T, static_cast<int>(s->Fs / 64), d->sms,
                           ktile_per_partial_byte(d, s->bn2), M * s->H * 4, false);
    }
    const size_t need = slots > 1 ? round256(static_cast<size_t>(slots * M * s->H) * 4) : 0;
    Workspace w;
    TP_TRY(get_ws(&w, workspace, ws_bytes, need, st));
    CUtensorMap ma;
    TP_TRY(make_map(&ma, A, s->H, M, 1, s->H * 2, M * s->H * 2, 128));
    TP_TRY(rowpar_tc(s, d, ma, 0, M, slots, reinterpret_cast<float *>(w.ptr), Z, st));
  }
  return TP_OK;
}

size_t tp_block_workspace_bytes(tp_shards_t attn, tp_shards_t mlp, int64_t M, tp_variant_t v) {
  DevState *d = nullptr;
  if (!attn || !mlp || attn->kind != 1 || mlp->kind != 0 || M <= 0 || !valid_variant(v) ||
      dev_state(&d) != TP_OK)
    return 0;
  BlockPlan p;
  plan_block(attn, mlp, M, v, d, &p);
  return p.total();
}

tp_status_t tp_block_forward(tp_shards_t attn, tp_shards_t mlp, const void *X, int64_t M, int causal,
                             tp_variant_t v, float *out, float *h_out, void *workspace, size_t ws_bytes,
                             void *stream) {
  return block_forward_impl(attn, mlp, X, M, causal, v, out, h_out, workspace, ws_bytes,
                            static_cast<cudaStream_t>(stream));
}

size_t tp_attention_workspace_bytes(int64_t M, int n_heads, int head_dim) {
  (void)M;
  (void)n_heads;
  (void)head_dim;
  return 0;  // the kernel reads Q, K and V as they are
}

tp_status_t tp_attention_forward(const void *Q, const void *K, const void *V, int64_t M, int n_heads,
                                 int head_dim, int causal, void *O, int64_t ldo, void *workspace,
                                 size_t ws_bytes, void *stream) {
  if (M < 0 || n_heads <= 0 || head_dim <= 0) return TP_ERR_ARG;
  if (head_dim != kAttnHeadDim) return TP_ERR_UNSUPPORTED;
  if (M == 0) return TP_OK;
  if (M > (1LL << 24) || cdiv(M, 128) * n_heads >= (1LL << 31)) return TP_ERR_UNSUPPORTED;
  if (!Q || !K || !V || !O || !aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O))
    return TP_ERR_ARG;
  const int64_t width = static_cast<int64_t>(n_heads) * head_dim;
  if (ldo < width || ldo % 8 != 0) return TP_ERR_ARG;
  const size_t in_bytes = static_cast<size_t>(M * width) * 2;
  const size_t out_bytes = static_cast<size_t>((M - 1) * ldo + width) * 2;
  if (ranges_overlap(O, out_bytes, Q, in_bytes) || ranges_overlap(O, out_bytes, K, in_bytes) ||
      ranges_overlap(O, out_bytes, V, in_bytes))
    return TP_ERR_ARG;
  (void)workspace;
  (void)ws_bytes;
  DevState *d = nullptr;
  TP_TRY(dev_state(&d));
  return attention_core(d, Q, K, V, M, n_heads, causal, O, ldo, static_cast<cudaStream_t>(stream));
}

tp_status_t tp_partial_sum(const float *const *Zi, int T, int64_t n, float *Z, void *stream) {
  if (!Zi || T < 1 || T > kMaxShards || n < 0) return TP_ERR_ARG;
  if (n == 0) return TP_OK;
  if (!Z) return TP_ERR_ARG;
  for (int t = 0; t < T; ++t)
    if (!Zi[t]) return TP_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(Z) & 3u) != 0) return TP_ERR_ARG;
  const uintptr_t z0 = reinterpret_cast<uintptr_t>(Z), z1 = z0 + static_cast<uintptr_t>(n) * 4;
  for (int t = 0; t < T; ++t) {
    if ((reinterpret_cast<uintptr_t>(Zi[t]) & 3u) != 0) return TP_ERR_ARG;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(Zi[t]), a1 = a0 + static_cast<uintptr_t>(n) * 4;
    const bool overlap = a0 < z1 && z0 < a1;
    if (overlap && !(t == 0 && a0 == z0)) return TP_ERR_ARG;
  }
  DevState *d = nullptr;
  TP_TRY(dev_state(&d));
  return cuda_status(launch_shard_sum(Zi, T, n, Z, d->sms, static_cast<cudaStream_t>(stream)));
}


tp_status_t tp_reduce_scatter(const float *const *Zi, int T, int64_t n, float *const *out, void *stream) {
  if (!Zi || !out || T < 1 || T > kMaxShards || n < 0) return TP_ERR_ARG;
  if (n % T != 0) return TP_ERR_INDIVISIBLE;
  if (n == 0) return TP_OK;
  const size_t bytes = static_cast<size_t>(n) * 4, bb = bytes / T;
  for (int t = 0; t < T; ++t) {
    if (!Zi[t] || !out[t] || (reinterpret_cast<uintptr_t>(Zi[t]) & 3u) ||
        (reinterpret_cast<uintptr_t>(out[t]) & 3u))
      return TP_ERR_ARG;
  }
  for (int i = 0; i < T; ++i) {
    for (int t = 0; t < T; ++t)
      if (ranges_overlap(out[i], bb, Zi[t], bytes)) return TP_ERR_ARG;
    for (int j = i + 1; j < T; ++j)
      if (ranges_overlap(out[i], bb, out[j], bb)) return TP_ERR_ARG;
  }
  DevState *d = nullptr;
  TP_TRY(dev_state(&d));
  return cuda_status(launch_reduce_scatter(Zi, T, n, out, d->sms, static_cast<cudaStream_t>(stream)));
}

tp_status_t tp_all_gather(const void *const *parts, int T, int64_t n_per, int elem_bytes, void *out,
                          void *stream) {
  if (!parts || T < 1 || T > kMaxShards || n_per < 0 || elem_bytes < 1 || elem_bytes > 16)
    return TP_ERR_ARG;
  if (n_per == 0) return TP_OK;
  if (!out) return TP_ERR_ARG;
  const size_t bb = static_cast<size_t>(n_per) * static_cast<size_t>(elem_bytes);
  char *o = static_cast<char *>(out);
  for (int t = 0; t < T; ++t) {
    if (!parts[t]) return TP_ERR_ARG;
    const bool in_place = parts[t] == o + static_cast<size_t>(t) * bb;
    if (!in_place && ranges_overlap(parts[t], bb, out, bb * T)) return TP_ERR_ARG;
  }
  DevState *d = nullptr;
  TP_TRY(dev_state(&d));
  return cuda_status(launch_all_gather(parts, T, static_cast<long long>(bb), out, d->sms,
                                       static_cast<cudaStream_t>(stream)));
}

tp_status_t tp_partial_sum_bf16(const float *const *Zi, int T, int64_t n, void *Z, void *stream) {
  if (!Zi || T < 1 || T > kMaxShards || n < 0) return TP_ERR_ARG;
  if (n == 0) return TP_OK;
  if (!Z || (reinterpret_cast<uintptr_t>(Z) & 1u)) return TP_ERR_ARG;
  for (int t = 0; t < T; ++t) {
    if (!Zi[t] || (reinterpret_cast<uintptr_t>(Zi[t]) & 3u)) return TP_ERR_ARG;
    if (ranges_overlap(Zi[t], static_cast<size_t>(n) * 4, Z, static_cast<size_t>(n) * 2)) return TP_ERR_ARG;
  }
  DevState *d = nullptr;
  TP_TRY(dev_state(&d));
  return cuda_status(launch_shard_sum_bf16(Zi, T, n, Z, d->sms, static_cast<cudaStream_t>(stream)));
}

tp_status_t tp_last_device_status(void *stream) {
  DevState *d = nullptr;
  TP_TRY(dev_state(&d));
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TP_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, d->status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return TP_ERR_CUDA;
  if (word != 0 && cudaMemset(d->status, 0, sizeof word) != cudaSuccess) return TP_ERR_CUDA;
  if (word & kDevTimeout) return TP_ERR_TIMEOUT;
  if (word & kDevCheck) return TP_ERR_DEVICE_CHECK;
  return TP_OK;
}

}  // extern "C"
