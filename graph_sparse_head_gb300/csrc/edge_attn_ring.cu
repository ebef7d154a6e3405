// Instantiations of the ring edge kernel (edge_ring.cuh) for fp16
// intermediates with 16 channels a lane: 8, 16 or 32 lanes per row.
#include "edge_ring.cuh"

#include <mutex>
#include <set>
#include <map>

namespace pmha {
namespace stream {

int ring_blocks_per_sm(const void *kern, int threads, int smem)
{
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find({dev, kern});
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, (size_t)smem) != cudaSuccess) return 0;
    cache[{dev, kern}] = n;
    return n;
}

pmha_status launch_ring_f16(int lpe, bool wv, const Args &k, cudaStream_t s)
{
    switch (lpe) {
    case 8: return wv ? launch_ring<8, true, false>(k, s) : launch_ring<8, false, false>(k, s);
    case 16: return wv ? launch_ring<16, true, false>(k, s) : launch_ring<16, false, false>(k, s);
    case 32: return wv ? launch_ring<32, true, false>(k, s) : launch_ring<32, false, false>(k, s);
    default: return PMHA_ERR_UNSUPPORTED;
    }
}

}  // namespace stream
}  // namespace pmha
