// Instances of the attention kernel for head dim 128 (one translation unit per
// head dim so they compile in parallel).
#include "attn_kernel.cuh"

namespace bsv {

cudaError_t launch_attention_d128(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                 const AttnParams &p, bool online, int n_ctas, cudaStream_t s) {
    return online ? launch_fwd_instance<128, true>(tq, tk, tv, p, n_ctas, s)
                  : launch_fwd_instance<128, false>(tq, tk, tv, p, n_ctas, s);
}

cudaError_t configure_attention_d128() { return configure_instance<128>(); }

}  // namespace bsv
