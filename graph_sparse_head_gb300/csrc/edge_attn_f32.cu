// Instantiations of the streaming edge kernel for float32 layers: 4 or 8
// channels per lane, 2 to 32 lanes per row.
#include "edge_stream.cuh"

namespace pmha {
namespace stream {

pmha_status launch_f32(int cpl, int lpe, bool wv, const Args &k, long long slots, cudaStream_t s)
{
    if (cpl == 4) return wv ? launch_lpe<float, 4, true>(lpe, k, slots, s) : launch_lpe<float, 4, false>(lpe, k, slots, s);
    if (cpl == 8) return wv ? launch_lpe<float, 8, true>(lpe, k, slots, s) : launch_lpe<float, 8, false>(lpe, k, slots, s);
    return PMHA_ERR_UNSUPPORTED;
}

}  // namespace stream
}  // namespace pmha
