// Tensor-core cross-decoder attention over an e4m3 cache ("KV cache memory
// systems", "Quantized cache changes attention inputs"): instantiations of
// the kernels in attn_tc.cuh with one-byte pages and per-page K/V scales.
#include "attn_tc.cuh"

namespace yoco {

cudaError_t launch_attn_tc_e4m3(const CUtensorMap& mk, const CUtensorMap& mv,
                                const AttnParams& p, int D, int BS, int sms, cudaStream_t s) {
    if (D == 128) return launch_d<128, true>(mk, mv, p, BS, sms, s);
    return launch_d<256, true>(mk, mv, p, BS, sms, s);
}

}  // namespace yoco
