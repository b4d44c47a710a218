// gemv.cu -- the wkv projection for a few tokens (stage 3, T <= 8), with the
// row gather and dequantisation (stage 2) fused into the x staging.
//
// kv[t, o] = bf16_rne(sum_i x[t, i] * wkv[o, i]), f32 accumulation
// (`linear_bf16`, metrale_model_arch/deepseek_v41_ref/engram.rs).  At one
// token the projection is a pass over wkv (251.7 MB a layer at V4.1 shape),
// so this kernel is shaped for HBM bandwidth, as the pages choose a GEMV over
// a tiled GEMM at m = 1 (spark_model/layers/attn_v41.rs, `Kernels.gemv`).
//
// Grid: the layers' CTAs side by side; each CTA owns a contiguous block of
// wkv rows of one layer.  Prologue: the CTA gathers that layer's T * C table
// rows (fp8 codes x pow2 scale, or Q2_K blocks) straight into x [T, K] bf16 in
// shared memory -- the [T * C, head_dim] rows never touch HBM.  Main loop:
// each warp takes one wkv row at a time; lane l streams the row's 16-byte
// chunks l, l + 32, ... with U loads in flight, multiplies them by x from
// shared memory and keeps a per-lane f32 sum in chunk order; a butterfly
// shuffle reduction then gives the dot product.  The order is fixed, so the
// fused and the plain-x launches give identical bits.
#include "common.cuh"

namespace engram {

constexpr int kGemvThreads = 512;
constexpr int kGemvUnroll = 8;

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float dot8(const uint4 &w, const uint4 &x, float acc) {
    acc = fmaf(bf16_lo(w.x), bf16_lo(x.x), acc);
    acc = fmaf(bf16_hi(w.x), bf16_hi(x.x), acc);
    acc = fmaf(bf16_lo(w.y), bf16_lo(x.y), acc);
    acc = fmaf(bf16_hi(w.y), bf16_hi(x.y), acc);
    acc = fmaf(bf16_lo(w.z), bf16_lo(x.z), acc);
    acc = fmaf(bf16_hi(w.z), bf16_hi(x.z), acc);
    acc = fmaf(bf16_lo(w.w), bf16_lo(x.w), acc);
    acc = fmaf(bf16_hi(w.w), bf16_hi(x.w), acc);
    return acc;
}

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

// Work units: a row of wkv is split into parts of 256 chunks (2048 values);
// warps take (row, part) units round-robin, so every warp streams the same
// amount to within one part (whole rows would leave a warp 8 or 9 rows, the
// last round a third full).  Lane l of a unit sums chunks part*256 + l + 32u,
// u = 0..7, in that order; a butterfly gives the part's sum; the parts of a
// row are added in part order.  gemv_q2k_kernel follows the same order.
template <int T, bool HASH>
__global__ void __launch_bounds__(kGemvThreads, 2) gemv_kernel(const __grid_constant__ GemvArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem_raw);
    int64_t *s_ids = reinterpret_cast<int64_t *>(smem_raw + (size_t)T * a.K * 2);
    float *psum = reinterpret_cast<float *>(smem_raw + (size_t)T * a.K * 2 + (HASH ? (size_t)T * a.C * 8 : 0));
    const int ctas_per_layer = gridDim.x / a.L;
    const int li = blockIdx.x / ctas_per_layer;
    const int cta = blockIdx.x % ctas_per_layer;
    const GemvLayer &ly = a.layer[li];
    const int K = a.K, N = a.N;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = kGemvThreads / 32;
    const int rows_per_cta = (N + ctas_per_layer - 1) / ctas_per_layer;
    const int r0 = cta * rows_per_cta;
    const int r1 = min(N, r0 + rows_per_cta);
    const int chunks = K >> 3;
    constexpr int kPart = 32 * kGemvUnroll;
    const int P = (chunks + kPart - 1) / kPart;
    const int units = max(r1 - r0, 0) * P;

    // ---- the first unit of this warp needs nothing computed: start its loads
    //      before waiting on the previous grid -------------------------------
    int u = warp;
    uint4 wv[kGemvUnroll];
    bool prefetched = u < units;
    if (prefetched) {
        const uint4 *wrow = reinterpret_cast<const uint4 *>(ly.wkv + (size_t)(r0 + u / P) * K);
        const int base = (u % P) * kPart;
#pragma unroll
        for (int k = 0; k < kGemvUnroll; ++k) {
            const int j = base + k * 32 + lane;
            wv[k] = j < chunks ? ld_stream(wrow + j) : make_uint4(0, 0, 0, 0);
        }
    }
    if (a.pdl) {
        griddep_wait();          // ids, cache, workspace: ready once the previous grid is done
        griddep_launch();        // the gate may now launch and prefetch the highway
    }

    // ---- row ids: hashed here (one thread per id), or read; then x -----------
    const int64_t *ids = ly.ids;
    int64_t id_stride = a.id_stride;
    if (HASH) {
        hash_ids(a, T, li, cta, s_ids);
        __syncthreads();
        ids = s_ids;
        id_stride = a.C;
    }
    stage_x(a, ly, T, ids, id_stride, xs, K);
    __syncthreads();

    // ---- stream this CTA's wkv units --------------------------------------------
    const uint4 *xs4 = reinterpret_cast<const uint4 *>(xs);
    for (; u < units; u += nwarps) {
        const int rl = u / P, part = u % P;
        const uint4 *wrow = reinterpret_cast<const uint4 *>(ly.wkv + (size_t)(r0 + rl) * K);
        const int base = part * kPart;
        if (!prefetched) {
#pragma unroll
            for (int k = 0; k < kGemvUnroll; ++k) {
                const int j = base + k * 32 + lane;
                wv[k] = j < chunks ? ld_stream(wrow + j) : make_uint4(0, 0, 0, 0);
            }
        }
        prefetched = false;
        float acc[T];
#pragma unroll
        for (int t = 0; t < T; ++t) acc[t] = 0.0f;
#pragma unroll
        for (int k = 0; k < kGemvUnroll; ++k) {
            const int j = base + k * 32 + lane;
            if (j < chunks) {
#pragma unroll
                for (int t = 0; t < T; ++t) acc[t] = dot8(wv[k], xs4[t * chunks + j], acc[t]);
            }
        }
#pragma unroll
        for (int t = 0; t < T; ++t) {
            float v = acc[t];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
            if (lane == 0) psum[((size_t)rl * T + t) * P + part] = v;
        }
    }
    __syncthreads();
    for (int i = tid; i < (r1 - r0) * T; i += kGemvThreads) {
        const int rl = i / T, t = i % T;
        float v = psum[(size_t)i * P];
        for (int part = 1; part < P; ++part) v += psum[(size_t)i * P + part];
        ly.kv[(size_t)t * N + r0 + rl] = (uint16_t)f32_to_bf16_bits(v);
    }
}

// ---------------------------------------------------------------------------
// 2..8 tokens: the same stream of wkv through mma.sync m16n8k16 (bf16 in, f32
// accumulate).  With several tokens a CUDA-core dot product needs one
// shared-memory read of x per token for every 16 bytes of wkv, more
// shared-memory traffic than the SM can serve at HBM rate; one mma covers 16
// wkv rows x 16 k x 8 tokens, so the kernel stays HBM-bound.
//
// wkv is streamed by the bulk-copy engine, not through registers: one
// producer warp copies 16-row x 1536-wide pieces of the CTA's rows (3 KB
// contiguous a row) into a 4-stage shared-memory ring, each stage completing
// an mbarrier by its byte count; 16 MMA warps read the pieces from shared
// memory and hand each stage back through a second mbarrier.  x is loop
// invariant for a warp (its k blocks are the same in every row group), so it
// lives in registers: staged once through the ring's upper half, then loaded
// as mma B fragments.
//
// The dot product runs over k, so any permutation of k applied to both
// operands gives the same sum; lane (g = lane/4, q = lane%4) holds physical k
// 8q .. 8q+7 of each 32-wide k block: one 16-byte shared-memory read of rows
// g and g + 8 (ring rows padded by 64 bytes, so 8 lanes of a phase hit 8
// distinct 16-byte bank groups) and token g's x feed two mma instructions.
// ---------------------------------------------------------------------------
constexpr int kMmaT = 8;
constexpr int kMmaWarps = 16;                           // MMA warps; one more warp copies
constexpr int kMmaThreads = (kMmaWarps + 1) * 32;
constexpr int kMmaJ = 3;                                // 32-wide k blocks a warp per stage
constexpr int kStageKb = kMmaWarps * kMmaJ;             // 48 k blocks (1536 values) a stage
constexpr int kMmaSubMax = 4;                           // stages a 16-row group: K <= 6144
constexpr int kMmaStages = 4;
constexpr uint32_t kRowBytes = kStageKb * 64 + 64;      // one row's piece + bank padding
constexpr uint32_t kMmaStageBytes = 16 * kRowBytes;     // 50 176
constexpr uint32_t kRedBytes = 2 * kMmaWarps * 32 * 16; // partial tiles, double-buffered
constexpr size_t kMmaSmemBytes = (size_t)kMmaStages * kMmaStageBytes + kRedBytes + 2 * kMmaStages * 8 + 16;
static_assert((size_t)kFusedHashMaxIds * 8 <= kRedBytes, "hashed ids are staged in the partial buffer");
static_assert((size_t)kMmaT * (kMmaSubMax * kStageKb * 32 + 8) * 2 <= 2 * (size_t)kMmaStageBytes,
              "x is staged in the ring's upper half");

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

// One CTA per SM, each owning a contiguous run of 16-row groups of one layer.
// Stage i of the CTA is group grp0 + i / nsub, k blocks 48 (i % nsub) .. +47;
// MMA warp w takes k blocks 3w .. 3w + 2 of every stage, and the 16 partial
// 16 x 8 tiles of a group are summed in warp order through shared memory.
template <bool HASH>
__global__ void __launch_bounds__(kMmaThreads, 1) gemv_mma_kernel(const __grid_constant__ GemvArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int K = a.K, N = a.N, T = a.T;
    const int xstride = K + 8;
    const uint32_t ring = smem_u32(smem_raw);
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem_raw + 2 * kMmaStageBytes);          // prologue only
    float *red = reinterpret_cast<float *>(smem_raw + kMmaStages * kMmaStageBytes);
    int64_t *s_ids = reinterpret_cast<int64_t *>(red);                                   // prologue only
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw + kMmaStages * kMmaStageBytes + kRedBytes);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * kMmaStages);
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int b) { return bar0 + 8u * b; };
    auto empty = [&](int b) { return bar0 + 8u * (kMmaStages + b); };

    const int ctas_per_layer = gridDim.x / a.L;
    const int li = blockIdx.x / ctas_per_layer;
    const int cta = blockIdx.x % ctas_per_layer;
    const GemvLayer &ly = a.layer[li];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int kblocks = K >> 5;
    const int nsub = (kblocks + kStageKb - 1) / kStageKb;                // <= kMmaSubMax (host-checked)
    const int groups_total = (N + 15) / 16;
    const int gpc = (groups_total + ctas_per_layer - 1) / ctas_per_layer;
    const int grp0 = cta * gpc, grp1 = min(groups_total, grp0 + gpc);
    const int ngroups = max(grp1 - grp0, 0);
    const int nstages = ngroups * nsub;
    const bool producer = warp == kMmaWarps;

    if (threadIdx.x == 0) {
        for (int b = 0; b < kMmaStages; ++b) {
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
    // Producer: stage i into slot i % 4 once the MMA warps have released it.
    auto issue_until = [&](int stop) {
        for (; issued < stop; ++issued) {
            const int i = issued, b = i % kMmaStages;
            bool ok = true;
            if (lane == 0) ok = mbar_wait(empty(b), ((i / kMmaStages) & 1) ^ 1, abort_flag, a.err);
            if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
            const int grp = grp0 + i / nsub, kb0 = (i % nsub) * kStageKb;
            const uint32_t bytes = (uint32_t)min(kStageKb, kblocks - kb0) * 64u;
            const int r0 = grp * 16, nrows = min(16, N - r0);
            if (lane == 0) mbar_expect_tx(full(b), bytes * (uint32_t)nrows);
            __syncwarp();
            if (lane < nrows)
                bulk_load(ring + b * kMmaStageBytes + lane * kRowBytes, ly.wkv + (size_t)(r0 + lane) * K + kb0 * 32,
                          bytes, full(b), pol);
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
    __syncthreads();                       // x is in registers: the ring's upper half is free

    if (producer) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // x staging writes before the copies
        issue_until(nstages);
        // Let every copy already issued land before the CTA can leave.
        if (lane == 0)
            for (int d = 1; d <= kMmaStages && issued - d >= 0; ++d) {
                const int i = issued - d;
                const uint64_t t0 = now_ns();
                while (!mbar_try(full(i % kMmaStages), (i / kMmaStages) & 1) && now_ns() - t0 < 10000000ull) {
                }
            }
        return;
    }

    bool live = true;
    const uint32_t a_off = g * kRowBytes + (warp * kMmaJ) * 64 + 16 * q;
    for (int gi = 0; gi < ngroups; ++gi) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int sub = 0; sub < kMmaSubMax; ++sub) {
            if (sub < nsub) {
                const int i = gi * nsub + sub, b = i % kMmaStages;
                const bool ok = live && mbar_wait(full(b), (i / kMmaStages) & 1, abort_flag, a.err);
                live = __all_sync(0xFFFFFFFFu, ok);
                if (live) {
                    const uint32_t sa = ring + b * kMmaStageBytes + a_off;
#pragma unroll
                    for (int jj = 0; jj < kMmaJ; ++jj) {
                        if (sub * kStageKb + warp * kMmaJ + jj < kblocks) {
                            const uint4 lo = lds128(sa + jj * 64), hi = lds128(sa + 8 * kRowBytes + jj * 64);
                            const uint4 xb = xr[sub][jj];
                            mma_16816(c, lo.x, hi.x, lo.y, hi.y, xb.x, xb.y);
                            mma_16816(c, lo.z, hi.z, lo.w, hi.w, xb.z, xb.w);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(empty(b));
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

template <bool HASH>
static cudaError_t launch_mma(const GemvArgs &a, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (a.T < 1 || a.T > kMmaT || a.K % 32 || (a.K >> 5) > kMmaSubMax * kStageKb) return cudaErrorInvalidValue;
    if (HASH && (size_t)a.T * a.C > (size_t)kFusedHashMaxIds) return cudaErrorInvalidValue;
    for (int l = 0; l < a.L; ++l)
        if (reinterpret_cast<uintptr_t>(a.layer[l].wkv) % 16) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gemv_mma_kernel<HASH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kMmaSmemBytes);
    if (e != cudaSuccess) return e;
    int ctas_per_layer = sms / a.L;
    const int groups = (a.N + 15) / 16;
    if (ctas_per_layer > groups) ctas_per_layer = groups;
    if (ctas_per_layer < 1) ctas_per_layer = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas_per_layer * a.L);
    cfg.blockDim = dim3(kMmaThreads);
    cfg.dynamicSmemBytes = kMmaSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_mma_kernel<HASH>, a);
}

// ---------------------------------------------------------------------------
// One token against Q2_K-quantised wkv ([N, K/256] blocks of 84 bytes, a row's
// blocks contiguous): `wkv_q2k` on spark_model/layers/engram_v41.rs, read by
// the single-token projection in place of the bf16 expansion, 6x fewer bytes.
// Lane l decodes weights 8l .. 8l+7 of every block -- exactly the k values it
// owns in gemv_kernel<1> (chunk 32 b + l) -- to bf16 and runs the same FMA
// sequence and the same butterfly, so kv is bit-identical to the bf16 GEMV on
// the dequantised weights.
// ---------------------------------------------------------------------------
constexpr int kQ2kUnroll = 8;     // blocks a unit: 8 x 256 values = one part of gemv_kernel<1>

// Small non-negative integer -> f32 without the quarter-rate conversion unit:
// 2^23 + n has n in its low mantissa bits, so subtracting 2^23 is exact.
__device__ __forceinline__ float small_u2f(uint32_t n) {
    return __uint_as_float(0x4B000000u | n) - 8388608.0f;
}

// Lane l's eight weights 8l .. 8l+7 of one Q2_K block, each rounded to bf16
// and widened back to f32 (the values the bf16 GEMV multiplies).  Same layout
// as q2k_lane_decode; y = fma(d*sc, q, -dmin*m) equals d*sc*q - dmin*m rounded
// once because d*sc*q is exact in f32.
__device__ __forceinline__ void q2k_lane_weights(uint32_t word, int lane, float (&w)[8]) {
    const int half = lane >> 4, j = (lane & 15) >> 2, m = lane & 3;
    const int qw = 4 + 8 * half + 2 * m;
    const uint32_t q0 = __shfl_sync(0xFFFFFFFFu, word, qw);
    const uint32_t q1 = __shfl_sync(0xFFFFFFFFu, word, qw + 1);
    const int sb = 8 * half + 2 * j + (m >> 1);
    const uint32_t scw = __shfl_sync(0xFFFFFFFFu, word, sb >> 2);
    const uint32_t dw = __shfl_sync(0xFFFFFFFFu, word, 20);
    const uint32_t sc = (scw >> (8 * (sb & 3))) & 0xFFu;
    const float d = __half2float(__ushort_as_half((unsigned short)(dw & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(dw >> 16)));
    const float dl = __fmul_rn(d, small_u2f(sc & 15u));
    const float nml = -__fmul_rn(dmin, small_u2f(sc >> 4));
    const uint32_t t0 = (q0 >> (2 * j)) & 0x03030303u, t1 = (q1 >> (2 * j)) & 0x03030303u;
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const uint32_t t = e < 4 ? t0 : t1;
        // byte e of t into the low byte of 0x4B000000: the f32 2^23 + q, minus 2^23
        const float f0 = __uint_as_float(__byte_perm(t, 0x4B000000u, 0x7540u | (e & 3))) - 8388608.0f;
        const float f1 = __uint_as_float(__byte_perm(t, 0x4B000000u, 0x7540u | ((e + 1) & 3))) - 8388608.0f;
        const float y0 = __fmaf_rn(dl, f0, nml);
        const float y1 = __fmaf_rn(dl, f1, nml);
        const uint32_t p = pack_bf16x2(y0, y1);
        w[e] = bf16_lo(p);
        w[e + 1] = bf16_hi(p);
    }
}

// A warp takes whole rows (round-robin); within a row it walks the parts of
// gemv_kernel<1> (8 blocks = 256 chunks each), loading part p + 1 while part
// p decodes, reduces each part by butterfly and adds the parts in order --
// the bf16 kernel's summation exactly, hence bit-identical kv.
template <bool HASH>
__global__ void __launch_bounds__(kGemvThreads, 2) gemv_q2k_kernel(const __grid_constant__ GemvArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    float *xf = reinterpret_cast<float *>(smem_raw);                       // x widened to f32 [K]
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem_raw + (size_t)a.K * 4);
    int64_t *s_ids = reinterpret_cast<int64_t *>(smem_raw + (size_t)a.K * 6);
    const int ctas_per_layer = gridDim.x / a.L;
    const int li = blockIdx.x / ctas_per_layer;
    const int cta = blockIdx.x % ctas_per_layer;
    const GemvLayer &ly = a.layer[li];
    const int K = a.K, N = a.N, nblk = K >> 8;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = kGemvThreads / 32;
    const int rows_per_cta = (N + ctas_per_layer - 1) / ctas_per_layer;
    const int r0 = cta * rows_per_cta;
    const int r1 = min(N, r0 + rows_per_cta);
    const int P = (nblk + kQ2kUnroll - 1) / kQ2kUnroll;

    auto load_part = [&](int o, int part, uint32_t (&dst)[kQ2kUnroll]) {
        const int bb = part * kQ2kUnroll;
        const uint32_t *w = reinterpret_cast<const uint32_t *>(ly.wkv_q2k + (size_t)o * nblk * 84) + lane;
#pragma unroll
        for (int k = 0; k < kQ2kUnroll; ++k) dst[k] = (bb + k < nblk && lane < 21) ? __ldg(w + 21 * (bb + k)) : 0u;
    };
    int o = r0 + warp;
    uint32_t wq[kQ2kUnroll];
    if (o < r1) load_part(o, 0, wq);
    if (a.pdl) {
        griddep_wait();
        griddep_launch();
    }
    const int64_t *ids = ly.ids;
    int64_t id_stride = a.id_stride;
    if (HASH) {
        hash_ids(a, 1, li, cta, s_ids);
        __syncthreads();
        ids = s_ids;
        id_stride = a.C;
    }
    stage_x(a, ly, 1, ids, id_stride, xs, K);
    __syncthreads();
    for (int i = tid; i < K / 2; i += kGemvThreads) {
        const uint32_t v = reinterpret_cast<const uint32_t *>(xs)[i];
        reinterpret_cast<float2 *>(xf)[i] = make_float2(bf16_lo(v), bf16_hi(v));
    }
    __syncthreads();

    const float4 *xf4 = reinterpret_cast<const float4 *>(xf);
    for (; o < r1; o += nwarps) {
        float row_sum = 0.0f;
        for (int part = 0; part < P; ++part) {
            // the next part (or the next row's first part) loads while this one decodes
            uint32_t wn[kQ2kUnroll];
            const bool more = part + 1 < P || o + nwarps < r1;
            if (part + 1 < P) load_part(o, part + 1, wn);
            else if (o + nwarps < r1) load_part(o + nwarps, 0, wn);
            const int b0 = part * kQ2kUnroll;
            float acc = 0.0f;
#pragma unroll
            for (int k = 0; k < kQ2kUnroll; ++k) {
                if (b0 + k < nblk) {                     // warp-uniform
                    float wv[8];
                    q2k_lane_weights(wq[k], lane, wv);
                    const int c = (b0 + k) * 32 + lane;  // the lane's 8 k values: chunk 32 b + l
                    const float4 xa = xf4[2 * c], xb = xf4[2 * c + 1];
                    acc = fmaf(wv[0], xa.x, acc);
                    acc = fmaf(wv[1], xa.y, acc);
                    acc = fmaf(wv[2], xa.z, acc);
                    acc = fmaf(wv[3], xa.w, acc);
                    acc = fmaf(wv[4], xb.x, acc);
                    acc = fmaf(wv[5], xb.y, acc);
                    acc = fmaf(wv[6], xb.z, acc);
                    acc = fmaf(wv[7], xb.w, acc);
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
            row_sum = part == 0 ? acc : row_sum + acc;
            if (more) {
#pragma unroll
                for (int k = 0; k < kQ2kUnroll; ++k) wq[k] = wn[k];
            }
        }
        if (lane == 0) ly.kv[o] = (uint16_t)f32_to_bf16_bits(row_sum);
    }
}

// Per-row part sums of one CTA: rows_per_cta x T x parts f32.
static size_t gemv_psum_bytes(int T, int K, int N, int ctas_per_layer) {
    const int P = ((K >> 3) + 32 * kGemvUnroll - 1) / (32 * kGemvUnroll);
    const int rows = (N + ctas_per_layer - 1) / ctas_per_layer;
    return (size_t)rows * T * P * 4;
}

template <bool HASH>
static cudaError_t launch_q2k_h(const GemvArgs &a, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int ctas_per_layer = (sms * 2) / a.L;
    const int max_useful = (a.N + 15) / 16;
    if (ctas_per_layer > max_useful) ctas_per_layer = max_useful;
    if (ctas_per_layer < 1) ctas_per_layer = 1;
    const size_t smem = (size_t)a.K * 6 + (HASH ? (size_t)a.C * 8 : 0);
    if (smem > 100 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gemv_q2k_kernel<HASH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas_per_layer * a.L);
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_q2k_kernel<HASH>, a);
}

cudaError_t launch_gemv_q2k(const GemvArgs &a, cudaStream_t s) {
    if (a.T != 1 || a.K % 256) return cudaErrorInvalidValue;
    return a.fuse_hash ? launch_q2k_h<true>(a, s) : launch_q2k_h<false>(a, s);
}

size_t gemv_smem_bytes(int T, int K) {
    if (T <= 1) {
        const size_t b = (size_t)K * 2 + (size_t)kFusedHashMaxIds * 8;
        return b <= 96 * 1024 ? b : SIZE_MAX;           // the rest of 100 KB holds part sums
    }
    if (T > kMmaT || K % 32 || (K >> 5) > kMmaSubMax * kStageKb) return SIZE_MAX;   // GEMM path
    return kMmaSmemBytes;
}

template <int T, bool HASH>
static cudaError_t launch_th(const GemvArgs &a, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t base_smem = (size_t)T * a.K * 2 + (HASH ? (size_t)T * a.C * 8 : 0);
    // two CTAs an SM (the launch bounds), each owning a contiguous block of rows
    int ctas_per_layer = (sms * 2) / a.L;
    const int max_useful = (a.N + 15) / 16;          // at least 16 rows a CTA
    if (ctas_per_layer > max_useful) ctas_per_layer = max_useful;
    if (ctas_per_layer < 1) ctas_per_layer = 1;
    const size_t smem = base_smem + gemv_psum_bytes(T, a.K, a.N, ctas_per_layer);
    if (smem > 100 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<T, HASH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas_per_layer * a.L);
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<T, HASH>, a);
}

template <int T>
static cudaError_t launch_t(const GemvArgs &a, cudaStream_t s) {
    return a.fuse_hash ? launch_th<T, true>(a, s) : launch_th<T, false>(a, s);
}

cudaError_t launch_gemv(const GemvArgs &a, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    if (a.T == 1) return launch_t<1>(a, s);
    if (gemv_smem_bytes(a.T, a.K) != SIZE_MAX)
        return a.fuse_hash ? launch_mma<true>(a, s) : launch_mma<false>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace engram
