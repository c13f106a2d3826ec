// Instances of the attention kernel for head dim 64 (one translation unit per
// head dim so they compile in parallel).
#include "attn_kernel.cuh"

namespace bsv {

#define BSV_CASE(NN)                                                                 \
    case NN:                                                                         \
        return online ? launch_fwd_instance<64, NN, true>(tq, tk, tv, p, n_ctas, s)  \
                      : launch_fwd_instance<64, NN, false>(tq, tk, tv, p, n_ctas, s);

cudaError_t launch_attention_d64(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                 const AttnParams &p, int N, bool online, int n_ctas, cudaStream_t s) {
    switch (N) {
        BSV_CASE(16) BSV_CASE(32) BSV_CASE(48) BSV_CASE(64)
        BSV_CASE(80) BSV_CASE(96) BSV_CASE(112) BSV_CASE(128)
        default: return cudaErrorInvalidValue;
    }
}
#undef BSV_CASE

cudaError_t configure_attention_d64(int N) {
    switch (N) {
        case 16: return configure_instance<64, 16>();
        case 32: return configure_instance<64, 32>();
        case 48: return configure_instance<64, 48>();
        case 64: return configure_instance<64, 64>();
        case 80: return configure_instance<64, 80>();
        case 96: return configure_instance<64, 96>();
        case 112: return configure_instance<64, 112>();
        case 128: return configure_instance<64, 128>();
        default: return cudaErrorInvalidValue;
    }
}

size_t smem_attention_d64(int N) {
    switch (N) {
        case 16: return AttnCfg<64, 16>::SMEM;
        case 32: return AttnCfg<64, 32>::SMEM;
        case 48: return AttnCfg<64, 48>::SMEM;
        case 64: return AttnCfg<64, 64>::SMEM;
        case 80: return AttnCfg<64, 80>::SMEM;
        case 96: return AttnCfg<64, 96>::SMEM;
        case 112: return AttnCfg<64, 112>::SMEM;
        case 128: return AttnCfg<64, 128>::SMEM;
        default: return 0;
    }
}

}  // namespace bsv
