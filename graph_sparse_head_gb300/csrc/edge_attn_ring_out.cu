// Instantiations of the ring edge kernel with out_proj tasks in its queue
// (edge_ring.cuh, edge_out.cuh): fp16 intermediates, embed_dim 128 (8 lanes
// per row).
#include "edge_ring.cuh"

namespace pmha {
namespace stream {

pmha_status launch_ring_out_f16(int lpe, const Args &k, cudaStream_t s)
{
    switch (lpe) {
    case 8: return launch_ring<8, true, true>(k, s);
    default: return PMHA_ERR_UNSUPPORTED;
    }
}

}  // namespace stream
}  // namespace pmha
