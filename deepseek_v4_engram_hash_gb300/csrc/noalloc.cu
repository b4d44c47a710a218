// noalloc.cu -- engram_forward with its scratch in a fixed device array, for
// callers that cannot allocate device memory (see include/engram.h).
//
// The scratch lives in this file's __device__ array, so the library holds it
// on every GPU that loads it.  Host code cannot use the array's name as a
// device address: the address is looked up once per device with
// cudaGetSymbolAddress (on the first call, with that device current) and
// passed down as the forward's workspace.  No call here allocates.
#include "common.cuh"

#include <mutex>

namespace engram {
bool hasher_geometry(const engram_hasher *hs, engram_geom *g, int *batch);
}

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;   // 4 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64] = {};

}  // namespace

extern "C" int engram_forward_noalloc(engram_hasher *hs, const engram_layer *layers, const int32_t *d_ids,
                                      int32_t T, int64_t start_pos, float *d_h, float eps, uintptr_t stream) {
    engram_geom g;
    int batch = 0;
    if (!engram::hasher_geometry(hs, &g, &batch)) return ENGRAM_E_NULL;
    if (T < 0) return ENGRAM_E_INVALID;
    // No tokens: the same checks and the same no-op as engram_forward; no
    // scratch is touched.
    if ((int64_t)batch * T == 0) return engram_forward(hs, layers, d_ids, T, start_pos, d_h, eps, nullptr, 0, stream);
    const size_t need = engram_workspace_bytes(&g, (int64_t)batch * T);
    if (need == 0) return ENGRAM_E_INVALID;
    if (need > kNoAllocScratchBytes) return ENGRAM_E_NOALLOC_LIMIT;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ENGRAM_E_CUDA;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return ENGRAM_E_CUDA;
            g_noalloc_ptr[dev] = p;
        }
        scratch = g_noalloc_ptr[dev];
    }
    return engram_forward(hs, layers, d_ids, T, start_pos, d_h, eps, scratch, kNoAllocScratchBytes, stream);
}
