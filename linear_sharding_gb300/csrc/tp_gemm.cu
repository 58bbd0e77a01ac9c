// tp_gemm.cu - launches of the tensor-core GEMM (tp_gemm_impl.cuh) for the
// forward epilogues: activations fused into the column-parallel GEMM,
// float32 partials / accumulated outputs of the row-parallel GEMM, and the
// swapped-operand decode tile.
#include "tp_gemm_impl.cuh"

namespace tp {

using namespace gemm_impl;

cudaError_t launch_gemm(GemmCfg cfg, Epi epi, const CUtensorMap &mapA, const CUtensorMap &mapB,
                        const GemmArgs &args, int num_sms, cudaStream_t stream) {
  if (epi >= EPI_GELU_SAVE_BF16) return launch_gemm_train(cfg, epi, mapA, mapB, args, num_sms, stream);
  switch (cfg) {
    case CFG_N256:
      switch (epi) {
        case EPI_GELU_BF16: return launch_impl<256, EPI_GELU_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_SWIGLU_BF16: return launch_impl<256, EPI_SWIGLU_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_IDENT_BF16: return launch_impl<256, EPI_IDENT_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_F32: return launch_impl<256, EPI_F32>(mapA, mapB, args, num_sms, stream);
        default: break;
      }
      break;
    case CFG_N128:
      switch (epi) {
        case EPI_GELU_BF16: return launch_impl<128, EPI_GELU_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_IDENT_BF16: return launch_impl<128, EPI_IDENT_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_F32: return launch_impl<128, EPI_F32>(mapA, mapB, args, num_sms, stream);
        default: break;
      }
      break;
    case CFG_N16:
      if (epi == EPI_F32_T) return launch_impl<16, EPI_F32_T>(mapA, mapB, args, num_sms, stream);
      break;
    case CFG_PAIR_N256:
      switch (epi) {
        case EPI_GELU_BF16: return launch_pair<EPI_GELU_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_SWIGLU_BF16: return launch_pair<EPI_SWIGLU_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_IDENT_BF16: return launch_pair<EPI_IDENT_BF16>(mapA, mapB, args, num_sms, stream);
        case EPI_F32: return launch_pair<EPI_F32>(mapA, mapB, args, num_sms, stream);
        default: break;
      }
      break;
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_wide(Epi epi, const CUtensorMap &mapA, const CUtensorMap &mapB, const CUtensorMap &mapB2,
                             const CUtensorMap &mapBr, const GemmArgs &args, int num_sms, cudaStream_t stream) {
  // every tile two MMAs (256 columns, then 32 .. kWideMaxN - 256), the widths multiples of 32
  const int narrowest = args.wide_nb == args.wide_q ? args.wide_bn : args.wide_bn - 32;
  if (narrowest <= 256 || args.wide_bn > kWideMaxN || args.wide_bn % 32 != 0 || args.wide_nb < 1 ||
      args.wide_nb > args.wide_q || args.slots != 1)
    return cudaErrorInvalidValue;
  if (epi == EPI_F32) return launch_pair<EPI_F32, true>(mapA, mapB, args, num_sms, stream, &mapB2, &mapBr);
  if (epi == EPI_F32_RESID)
    return launch_pair<EPI_F32_RESID, true>(mapA, mapB, args, num_sms, stream, &mapB2, &mapBr);
  return cudaErrorInvalidValue;
}

}  // namespace tp
