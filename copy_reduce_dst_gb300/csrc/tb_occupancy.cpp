// Per-device kernel set-up and occupancy, cached: raises a kernel's dynamic
// shared-memory limit where it needs more than the default 48 KiB and
// returns how many CTAs of it fit on one SM.  Both are properties of the
// device the call runs on, so the cache is keyed by device too.  The limit
// only ever grows (to the largest size asked for on that device), so every
// size a kernel was checked at stays launchable.  Safe to call from several
// host threads.

#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "tb_internal.h"

namespace tb {

int resident_ctas(const void *kernel, int threads, size_t smem)
{
    static std::mutex lock;
    static std::map<std::tuple<int, const void *, int, size_t>, int> cache;
    static std::map<std::pair<int, const void *>, size_t> limit;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess)
        return 0;
    const auto key = std::make_tuple(device, kernel, threads, smem);
    std::lock_guard<std::mutex> hold(lock);
    auto it = cache.find(key);
    if (it != cache.end())
        return it->second;
    if (smem > 48 * 1024) {
        size_t &cur = limit[std::make_pair(device, kernel)];
        if (smem > cur) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem) != cudaSuccess)
                return 0;
            cur = smem;
        }
    }
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, threads, smem) !=
            cudaSuccess ||
        blocks < 1)
        return 0;
    cache[key] = blocks;
    return blocks;
}

}  // namespace tb
