// tp_gemm_train.cu - launches of the tensor-core GEMM (tp_gemm_impl.cuh) for
// the training epilogues (the column-parallel GEMM that also keeps its
// pre-activations for the backward pass; the backward GEMM dH = dZ W2^T with
// the activation's derivative fused into its epilogue) and for the
// transformer block (the head-major QKV projection, and the row-parallel
// projections with their residual adds fused); and for the weight gradients,
// which read both operands MN-major (EPI_F32_MN).
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

}  // namespace tp
