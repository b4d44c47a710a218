// rows.cu -- table row gather and dequantisation (stage 2), standalone.
//
// fp8: `regen_table` + `embed_rows` on metrale_model_arch/deepseek_v41_ref/engram.rs:
//   row(id)[d] = bf16_rne(e4m3(table[id, d]) * scales[id, d / blk]).
// Q2_K: `rows_from_q2k` on spark_model/layers/engram_v41.rs, one 84-byte
//   ggml super-block per 256-wide row.
//
// Layout: hd/16 consecutive threads own one row; each moves 16 fp8 codes
// with one 16-byte load and stores 16 bf16 with two 16-byte stores, so a warp
// reads whole rows as contiguous 128-byte lines (hd = 256: 2 rows a warp).
#include "common.cuh"

namespace engram {

// Indices are 32-bit (the launcher splits a call so that every launch's
// thread count fits); the thread -> (row, part) and row -> (token, column)
// splits are shifts when head_dim and scale_block are powers of two, else one
// 32-bit division each -- 64-bit divisions would cost more than the copy.
// One 16-byte piece a thread: four pieces a thread with their loads batched
// measured slower (fewer, longer waves over random rows).
__global__ void __launch_bounds__(256) rows_fp8_kernel(const RowsArgs a) {
    const uint32_t lpr = (uint32_t)a.hd >> 4;                 // threads per row
    const uint32_t C = (uint32_t)a.C;
    const uint32_t total = (uint32_t)a.n_tok * C * lpr;
    const uint32_t nblk = (uint32_t)(a.hd / a.blk);
    const bool pow2 = ((lpr & (lpr - 1)) | ((uint32_t)a.blk & ((uint32_t)a.blk - 1))) == 0;
    const int ls = __ffs((int)lpr) - 1, bs = __ffs(a.blk) - 1;
    for (uint32_t g = blockIdx.x * blockDim.x + threadIdx.x; g < total; g += gridDim.x * blockDim.x) {
        const uint32_t row = pow2 ? g >> ls : g / lpr;
        const uint32_t part = g - row * lpr;
        const uint32_t t = row / C, c = row - t * C;
        const int64_t id = a.ids[(int64_t)t * a.id_stride + c];
        uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
        if (id >= 0 && id < a.R) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(a.table + id * a.hd) + part);
            const uint32_t sb = pow2 ? (part << 4) >> bs : (part << 4) / (uint32_t)a.blk;
            const float sc = fp8_row_scale(a.scales, a.fmt, id * nblk + sb);
            e4m3x4_scaled_to_bf16(v.x, sc, o0.x, o0.y);
            e4m3x4_scaled_to_bf16(v.y, sc, o0.z, o0.w);
            e4m3x4_scaled_to_bf16(v.z, sc, o1.x, o1.y);
            e4m3x4_scaled_to_bf16(v.w, sc, o1.z, o1.w);
        } else {
            set_err(a.err, ENGRAM_E_ROW);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(a.out + (size_t)row * a.hd) + 2 * part;
        dst[0] = o0;
        dst[1] = o1;
    }
}

// Q2_K: one warp per row.  Lanes 0..20 load the block's 21 little-endian
// words (the block is 4-byte aligned: 84 = 4 * 21); lane l then decodes values
// 8l .. 8l+7 (q2k_lane_decode).
__global__ void __launch_bounds__(256) rows_q2k_kernel(const RowsArgs a) {
    const int lane = threadIdx.x & 31;
    const uint32_t C = (uint32_t)a.C;
    const uint32_t n_rows = (uint32_t)a.n_tok * C;
    const uint32_t warps = gridDim.x * (blockDim.x >> 5);
    for (uint32_t row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < n_rows; row += warps) {
        const uint32_t t = row / C, c = row - t * C;
        const int64_t id = a.ids[(int64_t)t * a.id_stride + c];
        const bool ok = id >= 0 && id < a.R;
        uint32_t word = 0;
        if (ok && lane < 21) word = __ldg(reinterpret_cast<const uint32_t *>(a.table + id * 84) + lane);
        uint4 o = q2k_lane_decode(word, lane);
        if (!ok) {
            o = make_uint4(0, 0, 0, 0);
            if (lane == 0) set_err(a.err, ENGRAM_E_ROW);
        }
        reinterpret_cast<uint4 *>(a.out + (size_t)row * 256)[lane] = o;
    }
}

static unsigned grid_for(int64_t threads_needed) {
    int64_t b = (threads_needed + 255) / 256;
    if (b > 152 * 64) b = 152 * 64;
    return (unsigned)(b < 1 ? 1 : b);
}

// Tokens a launch may take so that its thread count (tokens x C x threads a
// row) stays below 2^31; larger calls go in several launches.
static int64_t tokens_per_launch(const RowsArgs &a, int64_t threads_per_row) {
    const int64_t per_tok = (int64_t)a.C * threads_per_row;
    return per_tok > 0 ? ((int64_t)1 << 31) / per_tok - 1 : a.n_tok;
}

template <class Kernel>
static cudaError_t launch_split(const RowsArgs &a, int64_t threads_per_row, int per_thread, Kernel k,
                                cudaStream_t s) {
    const int64_t step = tokens_per_launch(a, threads_per_row);
    if (step < 1) return cudaErrorInvalidValue;
    for (int64_t t0 = 0; t0 < a.n_tok; t0 += step) {
        RowsArgs b = a;
        b.n_tok = a.n_tok - t0 < step ? a.n_tok - t0 : step;
        b.ids = a.ids + t0 * a.id_stride;
        b.out = a.out + t0 * a.C * (int64_t)a.hd;
        k<<<grid_for((b.n_tok * a.C * threads_per_row + per_thread - 1) / per_thread), 256, 0, s>>>(b);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_rows_fp8(const RowsArgs &a, cudaStream_t s) {
    if (a.n_tok * a.C == 0) return cudaSuccess;
    return launch_split(a, a.hd >> 4, 1, rows_fp8_kernel, s);
}

cudaError_t launch_rows_q2k(const RowsArgs &a, cudaStream_t s) {
    if (a.n_tok * a.C == 0) return cudaSuccess;
    return launch_split(a, 32, 1, rows_q2k_kernel, s);
}

}  // namespace engram
