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

__device__ __forceinline__ int64_t compress(const HashArgs &a, int b, int64_t s) {
    const int32_t id = a.ids[(int64_t)b * a.T + s];
    if (id < 0 || (int64_t)id >= a.vocab) {
        set_err(a.err, ENGRAM_E_TOKEN);
        return -1;                                  // treated as unmapped
    }
    return a.token_map[id];
}

__global__ void __launch_bounds__(256) hash_kernel(const HashArgs a) {
    const int C = (a.ng - 1) * a.H;
    const int64_t total = (int64_t)a.B * a.T * a.L * C;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int col = (int)(g % C);
        const int li = (int)((g / C) % a.L);
        const int64_t bs = g / ((int64_t)C * a.L);
        const int s = (int)(bs % a.T);
        const int b = (int)(bs / a.T);
        const int64_t pos = a.start_pos + s;
        const int n_top = col / a.H + 1;            // this column's n-gram reaches shift n_top

        int64_t tok[kMaxNgram];
        bool blocked = false;
        for (int shift = 0; shift <= n_top; ++shift) {
            int64_t src;
            if (pos < shift) {
                src = 0;                            // blocked below; value unused
            } else if (pos - shift >= a.start_pos) {
                src = compress(a, b, pos - shift - a.start_pos);
            } else {
                src = a.cache[(int64_t)b * a.max_seq + (pos - shift)];
            }
            blocked = blocked || pos < shift || src == -1;
            tok[shift] = blocked ? a.pad_id : src;
        }
        const int64_t *m = a.mult + (int64_t)li * a.ng;
        uint64_t rolling = (uint64_t)tok[0] * (uint64_t)m[0];
        for (int n = 1; n <= n_top; ++n) rolling ^= (uint64_t)tok[n] * (uint64_t)m[n];
        const int64_t p = a.primes[(int64_t)li * C + col];
        int64_t r = (int64_t)rolling % p;
        if (r < 0) r += p;
        a.out[g] = (int64_t)((uint64_t)r + (uint64_t)a.offsets[(int64_t)li * C + col]);

        if (li == 0 && col == 0) a.cache[(int64_t)b * a.max_seq + pos] = compress(a, b, s);
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
