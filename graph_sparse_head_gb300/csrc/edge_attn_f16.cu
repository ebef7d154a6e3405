// Instantiations of the streaming edge kernel for fp16 intermediates
// (bf16 layers): 8 or 16 channels per lane, 2 to 32 lanes per row.
#include "edge_stream.cuh"

namespace pmha {
namespace stream {

pmha_status launch_f16(int cpl, int lpe, bool wv, const Args &k, long long slots, cudaStream_t s)
{
    if (cpl == 8) return wv ? launch_lpe<__half, 8, true>(lpe, k, slots, s) : launch_lpe<__half, 8, false>(lpe, k, slots, s);
    if (cpl == 16)
        return wv ? launch_lpe<__half, 16, true>(lpe, k, slots, s) : launch_lpe<__half, 16, false>(lpe, k, slots, s);
    return PMHA_ERR_UNSUPPORTED;
}

}  // namespace stream
}  // namespace pmha
