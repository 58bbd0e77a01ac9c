// tp_internal.h - declarations shared by the C ABI (tp_api.cu) and the
// kernel files.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tp_mlp.h"

namespace tp {

// Bits of the per-device status word the kernels report into.
constexpr unsigned kDevTimeout = 1u;
constexpr unsigned kDevCheck = 2u;

// Epilogues of the tensor-core GEMM.
enum Epi : int {
  EPI_GELU_BF16 = 0,    // Y = bf16(GeLU(acc)), written to the per-shard Y buffers
  EPI_SWIGLU_BF16 = 1,  // accumulator columns [0, BN/2) gate, [BN/2, BN) up -> bf16(SiLU(g) u)
  EPI_IDENT_BF16 = 2,   // Y = bf16(acc)
  EPI_F32 = 3,          // out[slot][row][col] = acc (float32 partials or the final Z)
  EPI_F32_T = 4,        // swapped operands: acc[feature][token] -> out[slot][token][feature]
  // training (backward) epilogues, same column-to-shard mapping as the bf16 ones:
  EPI_GELU_SAVE_BF16 = 5,    // out = bf16(GeLU(acc)), out2 = bf16(acc) (the pre-activation)
  EPI_SWIGLU_SAVE_BF16 = 6,  // out = bf16(SiLU(g) u), out2 = bf16(g), out3 = bf16(u)
  EPI_DGELU_BF16 = 7,        // out = bf16(acc * GeLU'(aux)), aux = saved pre-activation
  EPI_DSWIGLU_BF16 = 8,      // out = bf16(acc u SiLU'(g)), out2 = bf16(acc SiLU(g)); aux = g, aux2 = u
  EPI_QKV_HEADS_BF16 = 9,    // out = bf16(acc) head-major: [3][n_heads][M][head_dim] (Q, K, V)
  EPI_F32_RESID = 10,        // one slot: out = acc (+ aux, float32) (+ aux2, bf16), same layout as out;
                             // with out2, also out2 = bf16(out) (a residual add fused into the GEMM)
  EPI_F32_MN = 11            // as EPI_F32, with both operands MN-major (the weight gradients, whose K
                             // is the token axis): A and B are [segments][K][MN per segment] in
                             // memory, read through 4-D maps (kMnPairBox); a_mn_seg / b_mn_seg are
                             // the MN rows per segment (0: one segment)
};

// Packed rows of a SwiGLU shard alternate 128 gate rows and 128 up rows, so
// one 256-row B tile (or two 128-row A tiles) carries matching gate/up columns.
constexpr int kSwigluGranule = 128;

// Work description of one tensor-core GEMM launch: D[m][n] = sum_k A[m][k] B[n][k]
// over units (slot, m-tile, n-tile).  The virtual K axis is `kt_total` tiles
// of 64, made of segments (shards) of `kt_per_seg` tiles.  A segmented
// operand (a_seg / b_seg = 1) is a 3-D tensor map [segments][rows][K per
// segment] and k-tile kt reads coordinate (kt % kt_per_seg * 64, row,
// kt / kt_per_seg); a flat operand (0) is [1][rows][K] and reads (kt * 64,
// row, 0); a k-tile-blocked operand (kKtileBlocked, the packed bf16 weights)
// is [k-tiles][rows][64] and reads (0, row, kt).  With EPI_F32_MN both operands
// are MN-major and k-tile kt reads, for each 128 rows of the tile, (0, kt * 64,
// (row % mn_seg) / 64, row / mn_seg) of a 4-D map (kMnPairBox).  Slot s covers k-tiles [s*kt_per_slot,
// min(kt_total, (s+1)*kt_per_slot)).
constexpr int kKtileBlocked = 2;

struct GemmArgs {
  int m_tiles, n_tiles, slots;
  int kt_total, kt_per_seg, kt_per_slot;
  int a_seg, b_seg;
  int a_mn_seg, b_mn_seg;  // EPI_F32_MN: MN rows per segment of A / B (0: one segment)
  int group_m;          // raster: m-tiles per group (L2 reuse of B tiles)
  int rows_valid;       // valid output rows along A (M, or features when swapped)
  int cols_valid;       // valid output columns along B (N, or tokens when swapped)
  void *out;
  long long ld_out;        // elements between output rows
  long long slot_stride;   // elements between slots (EPI_F32, EPI_F32_T)
  long long shard_stride;  // elements between per-shard Y buffers (bf16 epilogues)
  int shard_cols;          // output columns per shard (bf16 epilogues)
  unsigned int *status;
  unsigned long long wait_limit_ns;
  void *out2, *out3;        // extra outputs of the training epilogues (same layout as out)
  const void *aux, *aux2;   // saved activations read by the backward epilogues (same layout)
  int head_dim;             // EPI_QKV_HEADS_BF16: columns per head
  int n_heads;              // EPI_QKV_HEADS_BF16: heads over all shards
  // Wide row-parallel schedule (launch_gemm_wide): each 256-row block of the output is cut into
  // wide_q tiles, wide_nb of wide_bn columns and the others of wide_bn - 32; a cluster runs one
  // tile at a time.
  int wide_bn, wide_nb, wide_q;
};

// Largest column count of one wide tile (two MMAs per k-step: 256 columns, then the rest).
constexpr int kWideMaxN = 480;

// MN-major operands (EPI_F32_MN) are 4-D tensor maps: dims {64 MN elements, K
// (tokens), MN blocks of 64 per segment, segments}, byte strides {MN per
// segment x 2, 128, K x MN per segment x 2}, box {64, 64, kMnPairBox, 1}.
// One copy lands kMnPairBox 64 x 64 blocks, 8 KiB apart; both lie in one
// segment because segments (shard widths) and tile rows are multiples of 128.
constexpr int kMnPairBox = 2;

// Tile configurations the GEMM is instantiated for.
enum GemmCfg : int {
  CFG_N256 = 0,  // BM 128 x BN 256, prefill
  CFG_N128 = 1,  // BM 128 x BN 128, prefill when the shard width is not a multiple of 256
  CFG_N16 = 2,   // BM 128 x BN 16, decode (weights as A, tokens as B)
  CFG_PAIR_N256 = 3  // CTA pair (cta_group::2): 256 x 256 tile, m_tiles count 256 rows,
                     // B tensor map box 128 rows (each CTA loads half of the B tile)
};

// Tensor map for the TMA stores of a GEMM epilogue: elements of 2 (bf16) or 4
// (float32) bytes, dims {d0 (contiguous), d1, d2}, byte strides {s1, s2}, box
// {box0, box1, 1} (box0 x elem_bytes = 128), 128-byte swizzle.  False if the
// driver rejects it.
bool encode_store_map(CUtensorMap *m, const void *base, int elem_bytes, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t s1, uint64_t s2, uint32_t box0, uint32_t box1);

// Launch the tensor-core GEMM.  Returns cudaSuccess or the launch error.
cudaError_t launch_gemm(GemmCfg cfg, Epi epi, const CUtensorMap &mapA, const CUtensorMap &mapB,
                        const GemmArgs &args, int num_sms, cudaStream_t stream);
// The row-parallel GEMM with float32 output (epi EPI_F32 or EPI_F32_RESID, one slot) on the
// wide schedule of GemmArgs::wide_*: the tiles in rounds of the CTA pairs that fit on the GPU at
// once, one tile per pair at a time.  mapB is the k-tile-blocked B operand with a 128-row box;
// mapB2 the same tensor with a (wide_bn - 256) / 2-row box and mapBr one with a
// (wide_bn - 288) / 2-row box (the second B piece of a tile, per CTA).
cudaError_t launch_gemm_wide(Epi epi, const CUtensorMap &mapA, const CUtensorMap &mapB, const CUtensorMap &mapB2,
                             const CUtensorMap &mapBr, const GemmArgs &args, int num_sms, cudaStream_t stream);
// The training epilogues (EPI_*_SAVE_BF16, EPI_D*_BF16); launch_gemm forwards to it.
cudaError_t launch_gemm_train(GemmCfg cfg, Epi epi, const CUtensorMap &mapA, const CUtensorMap &mapB,
                              const GemmArgs &args, int num_sms, cudaStream_t stream);


// Fused attention core over `heads` independent heads of dimension 128:
// O_h[r] = sum over keys j (j <= r when causal, j < M) of
// softmax_j(q_r . k_j * scale) v_j, for every token r < M.  Q, K and V are
// head-major [heads][M][128] bf16 tensor maps (Q box 64 x 128 rows, K box
// 64 x attention_key_box_rows(), V box 64 x 64 rows; rows past M read as
// zeros); O is bf16 [M][ldo] with head h in columns [128 h, 128 h + 128).
struct AttnArgs {
  int M;
  int heads;
  int m_tiles;        // key tiles of 128, ceil(M / 128)
  int causal;
  float scale_log2;   // scale * log2(e)
  void *O;
  long long ldo;
  unsigned int *status;
  unsigned long long wait_limit_ns;
};
constexpr int kAttnHeadDim = 128;
// Rows (keys) of the K tensor map's box: one 128-key tile per copy.
int attention_key_box_rows();
cudaError_t launch_attention(const CUtensorMap &mapQ, const CUtensorMap &mapK, const CUtensorMap &mapV,
                             const AttnArgs &args, int num_sms, cudaStream_t stream);

// Float32 CUDA-core GEMM: D[m][n] = sum_k A[m][k] B[n][k], same work model
// as the tensor-core path but with plain row-major pointers.  A rows have
// stride lda; segments (shards) of A and B along K are `a_seg`/`b_seg`
// elements apart; K per segment is `k_seg`, `segs_per_slot` segments per
// output slot.
struct SimtArgs {
  const float *A;
  const float *B;
  long long lda, ldb, a_seg, b_seg;
  int M, N, k_seg, nseg, segs_per_slot;
  int epi;              // EPI_GELU_BF16/EPI_SWIGLU_BF16/EPI_IDENT_BF16 write float32 here
  float *out;
  long long ld_out, slot_stride, shard_stride;
  int shard_cols;
};
cudaError_t launch_simt_gemm(const SimtArgs &a, cudaStream_t stream);

// Z[k] = sum over i ascending of P_i[k] (float32).
cudaError_t launch_shard_sum(const float *const *parts, int T, long long n, float *Z, int num_sms,
                             cudaStream_t stream);

// Shard-sum of `slots` float32 partials laid out `slot_stride` apart.
cudaError_t launch_shard_sum_strided(const float *P, int slots, long long slot_stride, long long n,
                                     float *Z, int num_sms, cudaStream_t stream);

// Reduce-scatter: out[i][k] = sum over t ascending of parts[t][i n/T + k].
cudaError_t launch_reduce_scatter(const float *const *parts, int T, long long n, float *const *out,
                                  int num_sms, cudaStream_t stream);
// All-gather: out = parts[0] | parts[1] | ... (nb_bytes each); a part already
// at its place in `out` is left alone.
cudaError_t launch_all_gather(const void *const *parts, int T, long long nb_bytes, void *out,
                              int num_sms, cudaStream_t stream);
// Shard-sum rounded once to bfloat16.
cudaError_t launch_shard_sum_bf16(const float *const *parts, int T, long long n, void *Z, int num_sms,
                                  cudaStream_t stream);

// h = x + z (x bf16, z float32) -> h float32 and hb = bf16(h).
cudaError_t launch_residual(const void *x, const float *z, float *h, void *hb, long long n, int num_sms,
                            cudaStream_t stream);
// out += h (float32).
cudaError_t launch_add_inplace(float *out, const float *h, long long n, int num_sms, cudaStream_t stream);

// Packing of weights into the K-major per-shard layout.
enum PackMode : int {
  PACK_W1 = 0,         // dst[s][r][k] = W1[k][s*Fs + r]
  PACK_W1_SWIGLU = 1,  // dst[s][r][k] = W1[k][gate/up column of packed row r]
  PACK_QKV = 2,        // dst[s][r][k] = Wqkv[k][(r / W) * H + s*W + r % W]
  PACK_ROWS = 3        // dst[s][n][k] = W2[s*Ks + k][n]
};
// Logical dst is [S][R][K]; src is row-major with leading dimension src_ld;
// esize is 2 or 4 bytes; `F` is the width of one half of [Wg | Wu], `H` the
// QKV hidden size, `W` the per-shard width (Fs or head columns).  Float32
// weights (CUDA-core path) are stored as [S][R][K].  Bfloat16 weights (TMA
// path, K a multiple of 64) are stored in k-tiles of 64, each tile holding
// the 64 K values of every row contiguously (see packed_index), so that one
// 128-row x 64 copy is one contiguous 16 KiB block of memory.
cudaError_t launch_pack(PackMode mode, const void *src, long long src_ld, void *dst, int S,
                        long long R, long long K, int esize, long long F, long long H, long long W,
                        cudaStream_t stream);
// Inverse: the logical shard s of S (row-major [H x W] for W1-like modes and
// `which` = 0/1 gate/up; [W x N] for PACK_ROWS) from the packed buffer.
cudaError_t launch_unpack(PackMode mode, const void *packed, void *dst, int s, int S, int which,
                          long long R, long long K, int esize, long long W, cudaStream_t stream);

// Decode finalize: h[s][t][j] = bf16(act(sum over slots of P[slot][t][row(s, j)])) for
// SwiGLU (gate and up rows) or GeLU/identity.
cudaError_t launch_decode_act(const float *P, int slots, long long slot_stride, long long ldp,
                              int M, int T, int Fs, int act, bool swiglu_rows, void *h,
                              cudaStream_t stream);

// True when `s` was made on the current device and that device's library
// state already exists (checked without creating it, so without allocating).
bool handle_ready_on_current_device(const tp_shards *s);

// The AUTO MLP plan fitted to a workspace of `budget` bytes: as tp_mlp_workspace_bytes(s, M,
// AUTO) when that fits; else the plan with no second-layer partials and, for decode, as many
// first-layer split-K slots as fit.  mlp_workspace_within returns its workspace bytes (0 on a
// bad argument; more than `budget` when even the smallest plan does not fit);
// mlp_forward_within runs it with `ws` (at least `budget` bytes) as the workspace.
size_t mlp_workspace_within(tp_shards *s, int64_t M, size_t budget);
tp_status_t mlp_forward_within(tp_shards *s, const void *X, int64_t M, tp_act_t act, float *Z, void *ws,
                               size_t budget, cudaStream_t st);

}  // namespace tp
