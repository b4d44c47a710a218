// rows.cu -- table row gather and dequantisation (stage 2): the standalone
// row kernels (engram_rows_*), and the prefill kernels that hash (stage 1)
// and gather every layer's rows in one launch.
//
// fp8: page "metrale_model_arch/deepseek_v41_ref/engram.rs", module doc, item 2:
//   row(id)[d] = bf16_rne(e4m3(table[id, d]) * scales[id, d / blk]).
// Q2_K: page "spark_model/layers/engram_v41.rs", module doc, item 2: one 84-byte
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

// The id of global row `row` = (m L + l) C + col of a fused hash + gather
// launch, hashed by one lane: writes it to the workspace and, for
// (l, col) = (0, 0), the position's cache entry; li and xrow = m C + col give
// the row's layer and its row in that layer's x.  A row past the end, or a
// device position that does not fit the cache (ok false, ENGRAM_E_CAPACITY
// already raised), reads as id -1.
__device__ __forceinline__ int64_t fused_row_id(const HashRowsArgs &r, const HashArgs &h, bool ok, int64_t sp,
                                                uint32_t row, uint32_t &li, uint32_t &xrow) {
    const uint32_t C = (uint32_t)r.layer[0].C, LC = (uint32_t)r.L * C, T = (uint32_t)h.T;
    int64_t id = -1;
    li = 0;
    xrow = 0;
    if (row < (uint32_t)r.M * LC) {
        const uint32_t m = row / LC, j = row - m * LC;
        li = j / C;
        const uint32_t col = j - li * C;
        xrow = m * C + col;
        if (ok) {
            const uint32_t b = m / T, s = m - b * T;
            id = hash_one(h, sp, (int)b, (int)s, (int)li, (int)col);
            if (j == 0) h.cache[(int64_t)b * h.max_seq + sp + s] = hash_compress(h, (int)b, s);
        }
        h.out[row] = id;
    }
    return id;
}

// Hash and fp8 gather of every layer in one launch (the larger steps; the
// hash kernel above is then not launched).  Global row r = (m L + l) C + col,
// the hash output's order.  A warp takes RB consecutive rows (RB <= 32): lane
// i < RB hashes row base + i with hash_one, writes the id and, for
// (l, col) = (0, 0), the position's cache entry; then the warp gathers the RB
// rows, 32 / lpr a pass, each thread taking its row's id, layer and x row
// from the hashing lane by shuffles, the loads of kU passes issued before any
// conversion.  A device position that does not fit the cache (ENGRAM_E_CAPACITY
// already raised) reads as id -1: zero rows, no row error on top.
// head_dim / 16 and scale_block are powers of two, head_dim <= 512.
// Measured on two V4.1 layers at 4096 tokens (hash + both gathers, against
// 8 + 2 x 16 us for the hash kernel and two gathers): RB = 16, kU = 2 34.5 -
// 35.1 us; RB = 8 34.7 - 35.4; RB = 32 36.5 - 39.7 (kU = 4 43, kU = 1 43 - 48);
// RB = 16 with kU = 1 38, kU = 4 42; the row's first thread hashing alone
// (2 of 32 lanes busy) 57 - 70 us; the rows staged in shared memory by bulk
// copies, one or two 32-row buffers a warp, 39 - 54 us.
template <int kU, int RB>
__global__ void __launch_bounds__(256, 6) hash_rows_fp8_kernel(const __grid_constant__ HashRowsArgs r,
                                                            const __grid_constant__ HashArgs h) {
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t n_rows = (uint32_t)r.M * (uint32_t)r.L * (uint32_t)r.layer[0].C;
    const int32_t hd = r.layer[0].hd;
    const int ls = __ffs(hd >> 4) - 1, bs = __ffs(r.layer[0].blk) - 1;
    const uint32_t per = 32u >> ls;                          // rows a pass
    const uint32_t sub = lane >> ls, part = lane & ((1u << ls) - 1);
    const uint32_t sb = (part << 4) >> bs;                   // the thread's scale block in its row
    const int64_t nblk = hd >> bs;
    int *err = r.layer[0].err;
    griddep_launch();                 // the GEMM after this may start its set-up; it waits for x
    int64_t sp;
    const bool ok = hash_start(h, sp);
    const uint32_t warps = gridDim.x * (blockDim.x >> 5);
    for (uint32_t base = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RB; base < n_rows;
         base += warps * RB) {
        uint32_t li = 0, xrow = 0;
        int64_t id = -1;
        if (lane < (uint32_t)RB) id = fused_row_id(r, h, ok, sp, base + lane, li, xrow);
#pragma unroll 1
        for (uint32_t p0 = 0; p0 < (uint32_t)RB; p0 += per * kU) {
            uint4 v[kU];
            float sc[kU];
            uint32_t pl[kU], px[kU];
            bool live[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const uint32_t i = (p0 + u * per + sub) & 31;   // the row's hashing lane (< RB when live)
                const int64_t rid = __shfl_sync(0xFFFFFFFFu, id, i);
                pl[u] = __shfl_sync(0xFFFFFFFFu, li, i);
                px[u] = __shfl_sync(0xFFFFFFFFu, xrow, i);
                live[u] = p0 + u * per + sub < (uint32_t)RB && base + i < n_rows;
                const RowsArgs &a = r.layer[pl[u]];
                v[u] = make_uint4(0, 0, 0, 0);
                sc[u] = 0.0f;
                if (live[u] && rid >= 0 && rid < a.R) {
                    v[u] = __ldg(reinterpret_cast<const uint4 *>(a.table + rid * hd) + part);
                    sc[u] = fp8_row_scale(a.scales, a.fmt, rid * nblk + sb);
                } else if (live[u] && ok) {
                    set_err(err, ENGRAM_E_ROW);
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                if (!live[u]) continue;
                uint4 o0, o1;                                    // zero codes x zero scale: zero rows
                e4m3x4_scaled_to_bf16(v[u].x, sc[u], o0.x, o0.y);
                e4m3x4_scaled_to_bf16(v[u].y, sc[u], o0.z, o0.w);
                e4m3x4_scaled_to_bf16(v[u].z, sc[u], o1.x, o1.y);
                e4m3x4_scaled_to_bf16(v[u].w, sc[u], o1.z, o1.w);
                uint4 *dst = reinterpret_cast<uint4 *>(r.layer[pl[u]].out + (size_t)px[u] * hd) + 2 * part;
                dst[0] = o0;
                dst[1] = o1;
            }
        }
    }
}

// Hash and Q2_K gather of every layer in one launch: a warp takes RB
// consecutive rows (RB <= 32), lanes 0 .. RB-1 hash one each; then the warp
// decodes the RB rows one at a time as rows_q2k_kernel does (lanes 0..20 hold
// the block's words), the words of kU rows loaded before any decode.  With
// 84-byte rows the gather moves little data, so fewer rows a warp (more
// warps) hide more of the load latency.  Measured on two V4.1 layers at 512
// tokens (hash + gathers 23 us as two kernels): RB = 8 with kU = 8 12.7 -
// 13.0 us; RB 8, kU 4 13.6; RB 8, kU 2 14.1 - 14.7; RB 4 13.8; RB 16 16.6.
template <int RB, int kU>
__global__ void __launch_bounds__(256) hash_rows_q2k_kernel(const __grid_constant__ HashRowsArgs r,
                                                            const __grid_constant__ HashArgs h) {
    static_assert(RB % kU == 0 && RB <= 32, "RB rows in passes of kU");
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t n_rows = (uint32_t)r.M * (uint32_t)r.L * (uint32_t)r.layer[0].C;
    int *err = r.layer[0].err;
    griddep_launch();                 // the GEMM after this may start its set-up; it waits for x
    int64_t sp;
    const bool ok = hash_start(h, sp);
    const uint32_t warps = gridDim.x * (blockDim.x >> 5);
    for (uint32_t base = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RB; base < n_rows;
         base += warps * RB) {
        uint32_t li = 0, xrow = 0;
        int64_t id = -1;
        if (lane < (uint32_t)RB) id = fused_row_id(r, h, ok, sp, base + lane, li, xrow);
#pragma unroll 1
        for (int p0 = 0; p0 < RB; p0 += kU) {
            uint32_t word[kU], px[kU], pl[kU];
            bool live[kU], valid[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = p0 + u;                              // the row's hashing lane
                const int64_t rid = __shfl_sync(0xFFFFFFFFu, id, i);
                pl[u] = __shfl_sync(0xFFFFFFFFu, li, i);
                px[u] = __shfl_sync(0xFFFFFFFFu, xrow, i);
                live[u] = base + i < n_rows;
                const RowsArgs &a = r.layer[pl[u]];
                valid[u] = live[u] && rid >= 0 && rid < a.R;
                if (live[u] && !valid[u] && ok && lane == 0) set_err(err, ENGRAM_E_ROW);
                word[u] = valid[u] && lane < 21 ? __ldg(reinterpret_cast<const uint32_t *>(a.table + rid * 84) + lane)
                                                : 0u;
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                if (!live[u]) continue;                            // the same for the whole warp
                uint4 o = q2k_lane_decode(word[u], (int)lane);
                if (!valid[u]) o = make_uint4(0, 0, 0, 0);
                reinterpret_cast<uint4 *>(r.layer[pl[u]].out + (size_t)px[u] * 256)[lane] = o;
            }
        }
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

// fp8 (f32 or e8m0 scales) in every layer, head_dim / 16 and scale_block
// powers of two, head_dim <= 512; or Q2_K (head_dim 256) in every layer.
bool hash_rows_supported(const HashRowsArgs &a) {
    if (a.L < 1 || a.L > kMaxLayers || a.M < 1) return false;
    const RowsArgs &r0 = a.layer[0];
    if (r0.C < 1 || a.M * a.L * (int64_t)r0.C >= ((int64_t)1 << 30)) return false;
    bool fp8 = true, q2k = r0.hd == 256;
    for (int l = 0; l < a.L; ++l) {
        fp8 = fp8 && (a.layer[l].fmt == ENGRAM_FMT_FP8 || a.layer[l].fmt == ENGRAM_FMT_FP8_E8M0);
        q2k = q2k && a.layer[l].fmt == ENGRAM_FMT_Q2K;
    }
    if (q2k) return true;
    const int lpr = r0.hd >> 4;
    return fp8 && r0.hd % 16 == 0 && lpr >= 1 && lpr <= 32 && (lpr & (lpr - 1)) == 0 && r0.blk >= 1 &&
           (r0.blk & (r0.blk - 1)) == 0 && r0.hd % r0.blk == 0;
}

cudaError_t launch_hash_rows(const HashRowsArgs &a, const HashArgs &h, cudaStream_t s) {
    if (!hash_rows_supported(a)) return cudaErrorInvalidValue;
    const int64_t n_rows = a.M * a.L * a.layer[0].C;
    auto grid = [](int64_t warps) {
        const int64_t blocks = (warps + 7) / 8;
        return (unsigned)(blocks < 152 * 64 ? blocks : 152 * 64);
    };
    if (a.layer[0].fmt == ENGRAM_FMT_Q2K)
        hash_rows_q2k_kernel<8, 8><<<grid((n_rows + 7) / 8), 256, 0, s>>>(a, h);
    else
        hash_rows_fp8_kernel<2, 16><<<grid((n_rows + 15) / 16), 256, 0, s>>>(a, h);
    return cudaGetLastError();
}

cudaError_t launch_rows_q2k(const RowsArgs &a, cudaStream_t s) {
    if (a.n_tok * a.C == 0) return cudaSuccess;
    return launch_split(a, 32, 1, rows_q2k_kernel, s);
}

}  // namespace engram
