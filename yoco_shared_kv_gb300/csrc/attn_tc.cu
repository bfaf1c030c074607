// Tensor-core cross-decoder attention over a bf16 cache: launch plumbing
// and the instantiations of the kernels in attn_tc.cuh.
#include "attn_tc.cuh"

namespace yoco {
namespace {

// Workers (warps, or warp pairs) of the attention kernel for a shape.
template <bool F8, int NT, bool PR = false>
int nw_of(int D, int BS) {
    switch (D * 100 + BS) {
        case 6416: return TcShape<64, 16, F8, NT, PR>::WK;
        case 6432: return TcShape<64, 32, F8, NT, PR>::WK;
        case 12816: return TcShape<128, 16, F8, NT, PR>::WK;
        case 12832: return TcShape<128, 32, F8, NT, PR>::WK;
        case 25616: return TcShape<256, 16, F8, NT, PR>::WK;
        default: return TcShape<256, 32, F8, NT, PR>::WK;
    }
}

}  // namespace

int tc_ctas(int sms) { return sms < kMaxCtas ? sms : kMaxCtas; }

size_t tc_workspace_bytes(int sms, int H_kv, int G, int D, int BS, bool e4m3) {
    (void)H_kv;
    const int64_t ctas = tc_ctas(sms);
    auto need = [&](int nw, int vs) {
        return static_cast<size_t>(tc_plan_bytes(ctas, nw)) +
               static_cast<size_t>(tc_pieces(ctas, nw, vs)) * (static_cast<size_t>(D) * 4 + 8);
    };
    // Two 8-head tiles (one warp's, or a warp pair's) run for groups wider than
    // 8 and for cross rows grouped 16 virtual heads wide; one tile for the rest
    // (8 virtual heads at most). A partial slot holds one tile's heads.
    const int nw2 = e4m3 ? nw_of<true, 2>(D, BS) : nw_of<false, 2>(D, BS);
    // (the pair shape's workers; shapes without pair kernels have no fewer)
    const int nwp = e4m3 ? nw_of<true, 1, true>(D, BS) : nw_of<false, 1, true>(D, BS);
    size_t b = need(nw2 > nwp ? nw2 : nwp, 16);
    if (G <= 8) {
        const int nw1 = e4m3 ? nw_of<true, 1>(D, BS) : nw_of<false, 1>(D, BS);
        const size_t b1 = need(nw1, 8);
        if (b1 > b) b = b1;
    }
    return b;
}

cudaError_t launch_attn_tc(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p,
                           int D, int BS, int sms, cudaStream_t s) {
    switch (D) {
        case 64: return launch_d<64, false>(mk, mv, p, BS, sms, s);
        case 128: return launch_d<128, false>(mk, mv, p, BS, sms, s);
        default: return launch_d<256, false>(mk, mv, p, BS, sms, s);
    }
}

}  // namespace yoco
