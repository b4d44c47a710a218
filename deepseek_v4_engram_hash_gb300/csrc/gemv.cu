// gemv.cu -- the wkv projection for a few tokens (stage 3, 1 <= T <= 8), with
// the row gather and dequantisation (stage 2) fused into the x staging.
//
// kv[t, o] = bf16_rne(sum_i x[t, i] * wkv[o, i]), f32 accumulation
// (`linear_bf16`, metrale_model_arch/deepseek_v41_ref/engram.rs).  At a few
// tokens the projection is a pass over wkv (251.7 MB a layer at V4.1 shape),
// so this kernel is shaped for HBM bandwidth, as the pages choose a GEMV over
// a tiled GEMM at m = 1 (spark_model/layers/attn_v41.rs, `Kernels.gemv`).
//
// Grid: the layers' CTAs side by side, one an SM; each CTA owns a contiguous
// run of 16-row groups of one layer's wkv.  Prologue: the CTA gathers that
// layer's T * C table rows (fp8 codes x pow2 scale, or Q2_K blocks) straight
// into x [T, K] bf16 in shared memory -- the [T * C, head_dim] rows never
// touch HBM.  Main loop: a copy warp streams the CTA's wkv rows into a
// shared-memory ring with bulk copies; 16 MMA warps multiply them by x on
// mma.sync m16n8k16 (bf16 in, f32 accumulate).  wkv may also be held as Q2_K
// blocks (`wkv_q2k` on spark_model/layers/engram_v41.rs, 6x fewer bytes): the
// same kernel then copies the blocks and decodes each lane's weights into its
// mma fragments, in the same order, so kv is bit-identical to the bf16 path on
// the dequantised weights.
#include "common.cuh"

namespace engram {

// Q2_K decode of one 256-wide row by one warp into shared memory.
__device__ __forceinline__ void q2k_row_to_smem(const uint8_t *blk, bool ok, int lane,
                                                uint16_t *dst) {
    uint32_t word = 0;
    if (ok && lane < 21) word = __ldg(reinterpret_cast<const uint32_t *>(blk) + lane);
    uint4 o = q2k_lane_decode(word, lane);
    if (!ok) o = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4 *>(dst)[lane] = o;
}

// Stage x [T rows, K] bf16 into shared memory at `xs` with row stride `xstride`
// elements: from a plain x, or by gathering and dequantising the layer's
// table rows ids[t * id_stride + c].
__device__ __forceinline__ void stage_x(const GemvArgs &a, const GemvLayer &ly, int T, const int64_t *ids,
                                        int64_t id_stride, uint16_t *xs, int xstride) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x, nwarps = nthreads >> 5;
    const int K = a.K, n_ids = T * a.C;
    if (!a.gather) {
        const int cpr = K >> 3;                      // 16-byte chunks a row
        for (int i = tid; i < T * cpr; i += nthreads) {
            const int t = i / cpr, j = i % cpr;
            reinterpret_cast<uint4 *>(xs + (size_t)t * xstride)[j] =
                __ldg(reinterpret_cast<const uint4 *>(ly.x + (size_t)t * K) + j);
        }
    } else if (ly.fmt != ENGRAM_FMT_Q2K) {
        const int lpr = a.hd >> 4, nblk = a.hd / a.blk;
        for (int g = tid; g < n_ids * lpr; g += nthreads) {
            const int row = g / lpr, part = g % lpr;
            const int t = row / a.C, c = row % a.C;
            const int64_t id = ids[(int64_t)t * id_stride + c];
            uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
            if (id >= 0 && id < ly.rows) {
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(ly.table + id * a.hd) + part);
                const float sc = fp8_row_scale(ly.scales, ly.fmt, id * nblk + (part * 16) / a.blk);
                e4m3x4_scaled_to_bf16(v.x, sc, o0.x, o0.y);
                e4m3x4_scaled_to_bf16(v.y, sc, o0.z, o0.w);
                e4m3x4_scaled_to_bf16(v.z, sc, o1.x, o1.y);
                e4m3x4_scaled_to_bf16(v.w, sc, o1.z, o1.w);
            } else {
                set_err(a.err, ENGRAM_E_ROW);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(xs + (size_t)t * xstride + (size_t)c * a.hd) + 2 * part;
            dst[0] = o0;
            dst[1] = o1;
        }
    } else {
        for (int row = warp; row < n_ids; row += nwarps) {
            const int t = row / a.C, c = row % a.C;
            const int64_t id = ids[(int64_t)t * id_stride + c];
            const bool ok = id >= 0 && id < ly.rows;
            if (!ok && lane == 0) set_err(a.err, ENGRAM_E_ROW);
            q2k_row_to_smem(ly.table + (ok ? id : 0) * 84, ok, lane, xs + (size_t)t * xstride + (size_t)c * 256);
        }
    }
}

// Row ids of this CTA's layer for the T tokens of the call, hashed here (one
// thread per id) into s_ids; the CTAs with index 0 in each layer also write
// them to the workspace, and the very first CTA writes the cache.
__device__ __forceinline__ void hash_ids(const GemvArgs &a, int T, int li, int cta, int64_t *s_ids) {
    const HashArgs &h = a.hash;
    int64_t sp;
    const bool ok = hash_start(h, sp);       // a device position past the cache: ids read as -1 (rows 0)
    for (int j = threadIdx.x; j < T * a.C; j += blockDim.x) {
        const int m = j / a.C, col = j % a.C;
        const int b = m / h.T, s = m % h.T;
        const int64_t id = ok ? hash_one(h, sp, b, s, li, col) : -1;
        s_ids[j] = id;
        if (cta == 0) h.out[((int64_t)m * a.L + li) * a.C + col] = id;
        if (ok && cta == 0 && li == 0 && col == 0)
            h.cache[(int64_t)b * h.max_seq + sp + s] = hash_compress(h, b, s);
    }
}


// ---------------------------------------------------------------------------
// The ring.  With several tokens a CUDA-core dot product needs one
// shared-memory read of x per token for every 16 bytes of wkv, more
// shared-memory traffic than the SM can serve at HBM rate; one mma covers 16
// wkv rows x 16 k x 8 tokens, so the kernel stays HBM-bound (at one token the
// unused seven token columns cost nothing: the tensor pipe is idle anyway).
//
// bf16 wkv: the copy warp copies 16-row x 1536-wide pieces of the CTA's rows
// (3 KB contiguous a row) into a 4-stage ring, each stage completing an
// mbarrier by its byte count; the MMA warps read the pieces from shared memory
// and hand each stage back through a second mbarrier.  Q2_K wkv: a stage is a
// whole 16-row group (16 x K/256 blocks of 84 bytes, contiguous in memory: one
// copy), six stages.  x is loop invariant for a warp (its k blocks are the
// same in every row group), so it lives in registers: staged once through the
// ring's upper half, then loaded as mma B fragments.
//
// The dot product runs over k, so any permutation of k applied to both
// operands gives the same sum; lane (g = lane/4, q = lane%4) holds physical k
// 8q .. 8q+7 of each 32-wide k block: one 16-byte shared-memory read of rows
// g and g + 8 (bf16 ring rows padded by 64 bytes, so the 8 lanes of a phase
// hit distinct 16-byte bank groups) and token g's x feed two mma instructions.
// ---------------------------------------------------------------------------
constexpr int kMmaT = 8;
constexpr int kMmaWarps = 16;                           // MMA warps; one more warp copies
constexpr int kMmaThreads = (kMmaWarps + 1) * 32;
constexpr int kMmaJ = 3;                                // 32-wide k blocks a warp per stage
constexpr int kStageKb = kMmaWarps * kMmaJ;             // 48 k blocks (1536 values) a bf16 stage
constexpr int kMmaSubMax = 4;                           // bf16 stages a 16-row group
static_assert(kMmaSubMax * kStageKb * 32 == kGemvMaxK, "x fragments cover K");
constexpr uint32_t kRowBytes = kStageKb * 64 + 64;      // one row's piece + bank padding
constexpr uint32_t kRedBytes = 2 * kMmaWarps * 32 * 16; // partial tiles, double-buffered
static_assert((size_t)kFusedHashMaxIds * 8 <= kRedBytes, "hashed ids are staged in the partial buffer");

template <bool WQ2K>
struct Ring;
template <>
struct Ring<false> {
    static constexpr int kStages = 4;
    static constexpr uint32_t kStageBytes = 16 * kRowBytes;                   // 50 176
};
template <>
struct Ring<true> {
    static constexpr int kStages = 6;
    static constexpr uint32_t kStageBytes = 16 * (kGemvMaxK / 256) * 84;      // 32 256
};
template <bool WQ2K>
constexpr size_t ring_smem_bytes() {
    return (size_t)Ring<WQ2K>::kStages * Ring<WQ2K>::kStageBytes + kRedBytes + 2 * Ring<WQ2K>::kStages * 8 + 16;
}
static_assert((size_t)kMmaT * (kGemvMaxK + 8) * 2 <= 2 * (size_t)Ring<false>::kStageBytes &&
                  (size_t)kMmaT * (kGemvMaxK + 8) * 2 <= 4 * (size_t)Ring<true>::kStageBytes,
              "x is staged in the ring's upper stages");

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Contiguous global -> shared copy by the bulk-copy engine, completing `bytes`
// on the mbarrier (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                          uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// The 16 MMA warps only (the copy warp does not take part).
__device__ __forceinline__ void mma_warps_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(kMmaWarps * 32) : "memory");
}

// Small non-negative integer -> f32 without the quarter-rate conversion unit:
// 2^23 + n has n in its low mantissa bits, so subtracting 2^23 is exact.
__device__ __forceinline__ float small_u2f(uint32_t n) {
    return __uint_as_float(0x4B000000u | n) - 8388608.0f;
}

// Lane (g, q)'s A-fragment words for 32-wide k block kb of one Q2_K row in
// shared memory: values v = 32 (kb % 8) + 8q + e, e = 0..7, of block kb / 8,
// each rounded to bf16, packed in pairs (the words a bf16 row holds there).
// With kk = kb % 8 the values share half = kk / 4, j = kk % 4 and sub-block
// 8 half + 2j + q/2; their quant bytes are qs[32 half + 8q + e] (block words
// 4 + 8 half + 2q and the next) and the quant is (byte >> 2j) & 3.
// A value is y = d*sc*q - dmin*m rounded once (d*sc*q and dmin*m are exact in
// f32, so fma(d*sc, q, -dmin*m) is that), then bf16: with one sub-block the
// lane's eight values take one of four, v[q].  v[0..3] are built once and
// each pair (v[q_e], v[q_e+1]) is one byte permute of them, its selector
// nibbles 2q_e, 2q_e + 1, 2q_e+1, 2q_e+1 + 1 = h * 0x22 + 0x1010 for the
// two quant bytes h = q_e + 256 q_e+1.
__device__ __forceinline__ uint4 q2k_frag(const uint8_t *row, int kb, int q) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(row + (kb >> 3) * 84);
    const int kk = kb & 7, half = kk >> 2, j = kk & 3;
    const uint32_t q0 = w[4 + 8 * half + 2 * q], q1 = w[5 + 8 * half + 2 * q];
    const int sb = 8 * half + 2 * j + (q >> 1);
    const uint32_t sc = (w[sb >> 2] >> (8 * (sb & 3))) & 0xFFu;
    const uint32_t dw = w[20];
    const float d = __half2float(__ushort_as_half((unsigned short)(dw & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(dw >> 16)));
    const float dl = __fmul_rn(d, small_u2f(sc & 15u));
    const float nml = -__fmul_rn(dmin, small_u2f(sc >> 4));
    const uint32_t v01 = pack_bf16x2(__fmaf_rn(dl, 0.0f, nml), __fmaf_rn(dl, 1.0f, nml));
    const uint32_t v23 = pack_bf16x2(__fmaf_rn(dl, 2.0f, nml), __fmaf_rn(dl, 3.0f, nml));
    const uint32_t t0 = (q0 >> (2 * j)) & 0x03030303u, t1 = (q1 >> (2 * j)) & 0x03030303u;
    return make_uint4(__byte_perm(v01, v23, t0 * 0x22u + 0x1010u),
                      __byte_perm(v01, v23, (t0 >> 16) * 0x22u + 0x1010u),
                      __byte_perm(v01, v23, t1 * 0x22u + 0x1010u),
                      __byte_perm(v01, v23, (t1 >> 16) * 0x22u + 0x1010u));
}

// One CTA per SM, each owning a contiguous run of 16-row groups of one layer.
// MMA warp w takes k blocks 48 s + 3w + j (s = 0 .. nsub-1, j = 0..2) of
// every row group, in that order, and the 16 partial 16 x 8 tiles of a group
// are summed in warp order through shared memory; both weight formats follow
// this order exactly.  bf16: stage i is group grp0 + i / nsub, k blocks
// 48 (i % nsub) .. +47.  Q2_K: stage i is group grp0 + i.
template <bool HASH, bool WQ2K>
__global__ void __launch_bounds__(kMmaThreads, 1) gemv_mma_kernel(const __grid_constant__ GemvArgs a) {
    using R = Ring<WQ2K>;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int K = a.K, N = a.N, T = a.T;
    const int xstride = K + 8;
    const uint32_t ring = smem_u32(smem_raw);
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem_raw + 2 * R::kStageBytes);          // prologue only
    float *red = reinterpret_cast<float *>(smem_raw + R::kStages * R::kStageBytes);
    int64_t *s_ids = reinterpret_cast<int64_t *>(red);                                   // prologue only
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw + R::kStages * R::kStageBytes + kRedBytes);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * R::kStages);
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int b) { return bar0 + 8u * b; };
    auto empty = [&](int b) { return bar0 + 8u * (R::kStages + b); };

    const int ctas_per_layer = gridDim.x / a.L;
    const int li = blockIdx.x / ctas_per_layer;
    const int cta = blockIdx.x % ctas_per_layer;
    const GemvLayer &ly = a.layer[li];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int kblocks = K >> 5;
    const int nsub = (kblocks + kStageKb - 1) / kStageKb;                // <= kMmaSubMax (host-checked)
    const uint32_t q2k_row = (uint32_t)(K >> 8) * 84u;                  // bytes of a Q2_K row
    const int groups_total = (N + 15) / 16;
    const int gpc = (groups_total + ctas_per_layer - 1) / ctas_per_layer;
    const int grp0 = cta * gpc, grp1 = min(groups_total, grp0 + gpc);
    const int ngroups = max(grp1 - grp0, 0);
    const int spg = WQ2K ? 1 : nsub;                                     // stages a group
    const int nstages = ngroups * spg;
    const bool producer = warp == kMmaWarps;

    if (threadIdx.x == 0) {
        for (int b = 0; b < R::kStages; ++b) {
            mbar_init(full(b), 1);
            mbar_init(empty(b), kMmaWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    const uint64_t pol = l2_evict_first();
    int issued = 0;
    // Copy warp: stage i into slot i % kStages once the MMA warps have released it.
    auto issue_until = [&](int stop) {
        for (; issued < stop; ++issued) {
            const int i = issued, b = i % R::kStages;
            bool ok = true;
            if (lane == 0) ok = mbar_wait(empty(b), ((i / R::kStages) & 1) ^ 1, abort_flag, a.err);
            if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
            const uint32_t dst = ring + b * R::kStageBytes;
            if (WQ2K) {
                // the group's rows are contiguous: one copy of the 16-byte multiple,
                // the last 4..12 bytes (a short last group only) by plain stores
                const int r0 = (grp0 + i) * 16, nrows = min(16, N - r0);
                const uint32_t total = (uint32_t)nrows * q2k_row, bulk = total & ~15u;
                const uint8_t *src = ly.wkv_q2k + (size_t)r0 * q2k_row;
                if (lane < (int)(total - bulk) / 4)
                    reinterpret_cast<uint32_t *>(smem_raw + b * R::kStageBytes + bulk)[lane] =
                        __ldg(reinterpret_cast<const uint32_t *>(src + bulk) + lane);
                __syncwarp();
                if (lane == 0) {
                    mbar_expect_tx(full(b), bulk);
                    if (bulk) bulk_load(dst, src, bulk, full(b), pol);
                }
            } else {
                const int grp = grp0 + i / nsub, kb0 = (i % nsub) * kStageKb;
                const uint32_t bytes = (uint32_t)min(kStageKb, kblocks - kb0) * 64u;
                const int r0 = grp * 16, nrows = min(16, N - r0);
                if (lane == 0) mbar_expect_tx(full(b), bytes * (uint32_t)nrows);
                __syncwarp();
                if (lane < nrows)
                    bulk_load(dst + lane * kRowBytes, ly.wkv + (size_t)(r0 + lane) * K + kb0 * 32, bytes, full(b), pol);
            }
        }
    };
    // the first two stages need nothing computed and do not overlap x: before the wait
    if (producer) issue_until(min(nstages, 2));

    if (a.pdl) {
        griddep_wait();
        griddep_launch();
    }
    const int64_t *ids = ly.ids;
    int64_t id_stride = a.id_stride;
    if (HASH) {
        hash_ids(a, T, li, cta, s_ids);
        __syncthreads();
        ids = s_ids;
        id_stride = a.C;
    }
    stage_x(a, ly, T, ids, id_stride, xs, xstride);
    __syncthreads();

    uint4 xr[kMmaSubMax][kMmaJ];
#pragma unroll
    for (int sub = 0; sub < kMmaSubMax; ++sub)
#pragma unroll
        for (int jj = 0; jj < kMmaJ; ++jj) {
            const int kb = sub * kStageKb + warp * kMmaJ + jj;
            xr[sub][jj] = (!producer && g < T && sub < nsub && kb < kblocks)
                              ? *reinterpret_cast<const uint4 *>(xs + (size_t)g * xstride + kb * 32 + 8 * q)
                              : make_uint4(0, 0, 0, 0);
        }
    __syncthreads();                       // x is in registers: the ring's upper stages are free

    if (producer) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // x staging writes before the copies
        issue_until(nstages);
        // Let every copy already issued land before the CTA can leave.
        if (lane == 0)
            for (int d = 1; d <= R::kStages && issued - d >= 0; ++d) {
                const int i = issued - d;
                const uint64_t t0 = now_ns();
                while (!mbar_try(full(i % R::kStages), (i / R::kStages) & 1) && now_ns() - t0 < 10000000ull) {
                }
            }
        return;
    }

    bool live = true;
    // wait for stage i: false (for the whole warp) once the CTA is aborting
    auto acquire = [&](int i) {
        const bool ok = live && mbar_wait(full(i % R::kStages), (i / R::kStages) & 1, abort_flag, a.err);
        live = __all_sync(0xFFFFFFFFu, ok);
        return live;
    };
    auto release = [&](int i) {
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(i % R::kStages));
    };
    const uint32_t a_off = g * kRowBytes + (warp * kMmaJ) * 64 + 16 * q;
    for (int gi = 0; gi < ngroups; ++gi) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        if (WQ2K) {
            if (acquire(gi)) {
                const uint8_t *row_lo = smem_raw + (gi % R::kStages) * R::kStageBytes + g * q2k_row;
                const uint8_t *row_hi = row_lo + 8 * q2k_row;
#pragma unroll
                for (int sub = 0; sub < kMmaSubMax; ++sub) {
#pragma unroll
                    for (int jj = 0; jj < kMmaJ; ++jj) {
                        const int kb = sub * kStageKb + warp * kMmaJ + jj;
                        if (sub < nsub && kb < kblocks) {
                            const uint4 lo = q2k_frag(row_lo, kb, q), hi = q2k_frag(row_hi, kb, q);
                            const uint4 xb = xr[sub][jj];
                            mma_16816(c, lo.x, hi.x, lo.y, hi.y, xb.x, xb.y);
                            mma_16816(c, lo.z, hi.z, lo.w, hi.w, xb.z, xb.w);
                        }
                    }
                }
                release(gi);
            }
        } else {
#pragma unroll
            for (int sub = 0; sub < kMmaSubMax; ++sub) {
                if (sub < nsub) {
                    const int i = gi * nsub + sub;
                    if (acquire(i)) {
                        const uint32_t sa = ring + (i % R::kStages) * R::kStageBytes + a_off;
#pragma unroll
                        for (int jj = 0; jj < kMmaJ; ++jj) {
                            if (sub * kStageKb + warp * kMmaJ + jj < kblocks) {
                                const uint4 lo = lds128(sa + jj * 64), hi = lds128(sa + 8 * kRowBytes + jj * 64);
                                const uint4 xb = xr[sub][jj];
                                mma_16816(c, lo.x, hi.x, lo.y, hi.y, xb.x, xb.y);
                                mma_16816(c, lo.z, hi.z, lo.w, hi.w, xb.z, xb.w);
                            }
                        }
                        release(i);
                    }
                }
            }
        }
        // Partials alternate between two buffers: the barrier of group i + 1
        // also orders the reads of group i before the writes of group i + 2.
        float *rb = red + (gi & 1) * (kMmaWarps * 32 * 4);
        reinterpret_cast<float4 *>(rb)[warp * 32 + lane] = make_float4(c[0], c[1], c[2], c[3]);
        mma_warps_sync();
        if (threadIdx.x < 128 && live) {
            // output (lane l, component j): c0 (row g, token 2q), c1 (row g, 2q+1), c2/c3 row g + 8
            const int l = threadIdx.x >> 2, j = threadIdx.x & 3;
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kMmaWarps; ++w) v += rb[(w * 32 + l) * 4 + j];
            const int gg = l >> 2, qq = l & 3;
            const int r = (grp0 + gi) * 16 + gg + ((j & 2) ? 8 : 0), t = 2 * qq + (j & 1);
            if (r < N && t < T) ly.kv[(size_t)t * N + r] = (uint16_t)f32_to_bf16_bits(v);
        }
    }
}

template <bool HASH, bool WQ2K>
static cudaError_t launch_mma(const GemvArgs &a, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (a.T < 1 || a.T > kMmaT || a.K % (WQ2K ? 256 : 32) || a.K > kGemvMaxK) return cudaErrorInvalidValue;
    if (HASH && (size_t)a.T * a.C > (size_t)kFusedHashMaxIds) return cudaErrorInvalidValue;
    for (int l = 0; l < a.L; ++l) {
        const void *w = WQ2K ? static_cast<const void *>(a.layer[l].wkv_q2k) : static_cast<const void *>(a.layer[l].wkv);
        if (!w || reinterpret_cast<uintptr_t>(w) % 16) return cudaErrorInvalidValue;
    }
    const size_t smem = ring_smem_bytes<WQ2K>();
    cudaError_t e = cudaFuncSetAttribute(gemv_mma_kernel<HASH, WQ2K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    int ctas_per_layer = sms / a.L;
    const int groups = (a.N + 15) / 16;
    if (ctas_per_layer > groups) ctas_per_layer = groups;
    if (ctas_per_layer < 1) ctas_per_layer = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas_per_layer * a.L);
    cfg.blockDim = dim3(kMmaThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_mma_kernel<HASH, WQ2K>, a);
}

size_t gemv_smem_bytes(int T, int K) {
    if (T < 1 || T > kMmaT || K % 32 || K > kGemvMaxK) return SIZE_MAX;   // GEMM path
    return ring_smem_bytes<false>();
}

cudaError_t launch_gemv(const GemvArgs &a, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    return a.fuse_hash ? launch_mma<true, false>(a, s) : launch_mma<false, false>(a, s);
}

cudaError_t launch_gemv_q2k(const GemvArgs &a, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    return a.fuse_hash ? launch_mma<true, true>(a, s) : launch_mma<false, true>(a, s);
}

}  // namespace engram
