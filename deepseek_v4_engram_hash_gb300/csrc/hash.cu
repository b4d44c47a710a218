// hash.cu -- the n-gram hash (stage 1).
//
// Page "metrale_model_arch/deepseek_v41_ref/engram.rs", module doc, item 1 (and
// page "spark_model/layers/engram_v41.rs", module doc, item 1), batched: for position p = start_pos + s of sequence b, the window holds the
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

// 32-bit indices (the launcher splits larger calls by sequence): the split
// of a thread index into (token, layer, column) is two 32-bit divisions.
__global__ void __launch_bounds__(256) hash_kernel(const HashArgs a) {
    const uint32_t C = (uint32_t)((a.ng - 1) * a.H), LC = (uint32_t)a.L * C, T = (uint32_t)a.T;
    const uint32_t total = (uint32_t)a.B * T * LC;
    int64_t sp;
    if (!hash_start(a, sp)) return;
    for (uint32_t g = blockIdx.x * blockDim.x + threadIdx.x; g < total; g += gridDim.x * blockDim.x) {
        const uint32_t m = g / LC, j = g - m * LC;
        const uint32_t li = j / C, col = j - li * C;
        const uint32_t b = m / T, s = m - b * T;
        a.out[g] = hash_one(a, sp, (int)b, (int)s, (int)li, (int)col);
        if (j == 0) a.cache[(int64_t)b * a.max_seq + sp + s] = hash_compress(a, (int)b, s);
    }
}

cudaError_t launch_hash(const HashArgs &a, cudaStream_t s) {
    const int64_t per_seq = (int64_t)a.T * a.L * (a.ng - 1) * a.H;
    if (per_seq * a.B == 0) return cudaSuccess;
    if (per_seq >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
    const int64_t seqs = ((int64_t)1 << 31) / per_seq;               // sequences a launch
    for (int64_t b0 = 0; b0 < a.B; b0 += seqs) {
        HashArgs h = a;
        h.B = (int32_t)(a.B - b0 < seqs ? a.B - b0 : seqs);
        h.ids = a.ids + b0 * a.T;
        h.cache = a.cache + b0 * a.max_seq;
        h.out = a.out + b0 * per_seq;
        const int64_t blocks = (per_seq * h.B + 255) / 256;
        hash_kernel<<<(unsigned)(blocks < 65535 ? blocks : 65535), 256, 0, s>>>(h);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace engram
