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

__global__ void __launch_bounds__(256) rows_fp8_kernel(const RowsArgs a) {
    const int lpr = a.hd >> 4;                       // threads per row
    const int64_t n_rows = a.n_tok * a.C;
    const int nblk = a.hd / a.blk;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < n_rows * lpr;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = g / lpr;
        const int part = (int)(g % lpr);
        const int64_t t = row / a.C;
        const int c = (int)(row % a.C);
        const int64_t id = a.ids[t * a.id_stride + c];
        uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
        if (id >= 0 && id < a.R) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(a.table + id * a.hd) + part);
            const float sc = fp8_row_scale(a.scales, a.fmt, id * nblk + (part * 16) / a.blk);
            e4m3x4_scaled_to_bf16(v.x, sc, o0.x, o0.y);
            e4m3x4_scaled_to_bf16(v.y, sc, o0.z, o0.w);
            e4m3x4_scaled_to_bf16(v.z, sc, o1.x, o1.y);
            e4m3x4_scaled_to_bf16(v.w, sc, o1.z, o1.w);
        } else {
            set_err(a.err, ENGRAM_E_ROW);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(a.out + row * a.hd) + 2 * part;
        dst[0] = o0;
        dst[1] = o1;
    }
}

// Q2_K: one warp per row.  Lanes 0..20 load the block's 21 little-endian
// words (the block is 4-byte aligned: 84 = 4 * 21); lane l then decodes values
// 8l .. 8l+7 (q2k_lane_decode).
__global__ void __launch_bounds__(256) rows_q2k_kernel(const RowsArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t n_rows = a.n_tok * a.C;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < n_rows;
         row += warps) {
        const int64_t t = row / a.C;
        const int c = (int)(row % a.C);
        const int64_t id = a.ids[t * a.id_stride + c];
        const bool ok = id >= 0 && id < a.R;
        uint32_t word = 0;
        if (ok && lane < 21) word = __ldg(reinterpret_cast<const uint32_t *>(a.table + id * 84) + lane);
        uint4 o = q2k_lane_decode(word, lane);
        if (!ok) {
            o = make_uint4(0, 0, 0, 0);
            if (lane == 0) set_err(a.err, ENGRAM_E_ROW);
        }
        reinterpret_cast<uint4 *>(a.out + row * 256)[lane] = o;
    }
}

static unsigned grid_for(int64_t threads_needed) {
    int64_t b = (threads_needed + 255) / 256;
    if (b > 152 * 64) b = 152 * 64;
    return (unsigned)(b < 1 ? 1 : b);
}

cudaError_t launch_rows_fp8(const RowsArgs &a, cudaStream_t s) {
    const int64_t n = a.n_tok * a.C * (a.hd >> 4);
    if (n == 0) return cudaSuccess;
    rows_fp8_kernel<<<grid_for(n), 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_rows_q2k(const RowsArgs &a, cudaStream_t s) {
    const int64_t n = a.n_tok * a.C * 32;
    if (n == 0) return cudaSuccess;
    rows_q2k_kernel<<<grid_for(n), 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace engram
