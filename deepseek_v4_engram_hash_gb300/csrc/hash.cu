// hash.cu -- the n-gram hash (stage 1).
//
// `EngramHasher::hash` (spark_model/layers/engram_v41.rs) and
// `NgramHashState::forward` (metrale_model_arch/deepseek_v41_ref/engram.rs),
// batched: for position p = start_pos + s of sequence b, the window holds the
// compressed ids at shifts 0..ng-1; once a shift reaches before position 0 or
// an unmapped (-1) id, that shift and every larger one take pad_id.  Per layer,
// rolling = tok0 * m0, then rolling ^= tok_n * m_n for n = 1..ng-1, and column
// (n-1)*H + h = rem_euclid(rolling, prime) + offset.  i64 with wrap.
//
// One thread per (b, s, layer, column): 24 * 2 ids a token at V4.1 shape.
// The thread rebuilds its own window: ids of this call come straight from the
// input (through token_map), older positions from the cache, so no thread
// depends on another thread's cache write.  The (layer 0, column 0) thread
// of each position writes that position's compressed id into the cache.
#include "common.cuh"

namespace engram {

__global__ void __launch_bounds__(256) hash_kernel(const HashArgs a) {
    const int C = (a.ng - 1) * a.H;
    const int64_t total = (int64_t)a.B * a.T * a.L * C;
    int64_t sp;
    if (!hash_start(a, sp)) return;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int col = (int)(g % C);
        const int li = (int)((g / C) % a.L);
        const int64_t bs = g / ((int64_t)C * a.L);
        const int s = (int)(bs % a.T);
        const int b = (int)(bs / a.T);
        a.out[g] = hash_one(a, sp, b, s, li, col);
        if (li == 0 && col == 0) a.cache[(int64_t)b * a.max_seq + sp + s] = hash_compress(a, b, s);
    }
}

cudaError_t launch_hash(const HashArgs &a, cudaStream_t s) {
    const int C = (a.ng - 1) * a.H;
    const int64_t total = (int64_t)a.B * a.T * a.L * C;
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    hash_kernel<<<(unsigned)(blocks < 65535 ? blocks : 65535), threads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace engram
