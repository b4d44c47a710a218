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

// Q2_K decode of one 256-wide row by one warp (see rows.cu for the layout).
__device__ __forceinline__ void q2k_row_to_smem(const uint8_t *blk, bool ok, int lane,
                                                uint16_t *dst) {
    const int half = lane >> 4, j = (lane & 15) >> 2, m = lane & 3;
    uint32_t word = 0;
    if (ok && lane < 21) word = __ldg(reinterpret_cast<const uint32_t *>(blk) + lane);
    const int qw = 4 + 8 * half + 2 * m;
    const uint32_t q0 = __shfl_sync(0xFFFFFFFFu, word, qw);
    const uint32_t q1 = __shfl_sync(0xFFFFFFFFu, word, qw + 1);
    const int sb = 8 * half + 2 * j + (m >> 1);
    const uint32_t scw = __shfl_sync(0xFFFFFFFFu, word, sb >> 2);
    const uint32_t dw = __shfl_sync(0xFFFFFFFFu, word, 20);
    const uint32_t sc = (scw >> (8 * (sb & 3))) & 0xFFu;
    const float d = __half2float(__ushort_as_half((unsigned short)(dw & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(dw >> 16)));
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t byte = ((e < 4 ? q0 : q1) >> (8 * (e & 3))) & 0xFFu;
        y[e] = q2k_value(d, dmin, sc, (byte >> (2 * j)) & 3u);
    }
    uint4 o = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                         pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
    if (!ok) o = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4 *>(dst)[lane] = o;
}

template <int T, bool HASH>
__global__ void __launch_bounds__(kGemvThreads, 2) gemv_kernel(const __grid_constant__ GemvArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem_raw);
    int64_t *s_ids = reinterpret_cast<int64_t *>(smem_raw + (size_t)T * a.K * 2);
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

    // ---- the first batch of this warp's wkv stream needs nothing computed:
    //      start it before waiting on the previous grid ------------------------
    int o = r0 + warp;
    uint4 wv[kGemvUnroll];
    bool prefetched = o < r1;
    if (prefetched) {
        const uint4 *wrow = reinterpret_cast<const uint4 *>(ly.wkv + (size_t)o * K);
#pragma unroll
        for (int u = 0; u < kGemvUnroll; ++u) {
            const int j = u * 32 + lane;
            wv[u] = j < chunks ? ld_stream(wrow + j) : make_uint4(0, 0, 0, 0);
        }
    }
    if (a.pdl) {
        griddep_wait();          // ids, cache, workspace: ready once the previous grid is done
        griddep_launch();        // the gate may now launch and prefetch the highway
    }

    // ---- row ids: hashed here (one thread per id), or read ------------------
    const int n_ids = T * a.C;
    const int64_t *ids = ly.ids;
    int64_t id_stride = a.id_stride;
    if (HASH) {
        const HashArgs &h = a.hash;
        for (int j = tid; j < n_ids; j += kGemvThreads) {
            const int m = j / a.C, col = j % a.C;
            const int b = m / h.T, s = m % h.T;
            const int64_t id = hash_one(h, b, s, li, col);
            s_ids[j] = id;
            if (cta == 0) h.out[((int64_t)m * a.L + li) * a.C + col] = id;
            if (cta == 0 && li == 0 && col == 0)
                h.cache[(int64_t)b * h.max_seq + h.start_pos + s] = hash_compress(h, b, s);
        }
        __syncthreads();
        ids = s_ids;
        id_stride = a.C;
    }

    // ---- stage x [T, K] bf16 in shared memory --------------------------------
    if (!a.gather) {
        const uint4 *src = reinterpret_cast<const uint4 *>(ly.x);
        uint4 *dst = reinterpret_cast<uint4 *>(xs);
        for (int i = tid; i < T * K / 8; i += kGemvThreads) dst[i] = __ldg(src + i);
    } else if (ly.fmt == ENGRAM_FMT_FP8) {
        const int lpr = a.hd >> 4, nblk = a.hd / a.blk;
        for (int g = tid; g < n_ids * lpr; g += kGemvThreads) {
            const int row = g / lpr, part = g % lpr;
            const int t = row / a.C, c = row % a.C;
            const int64_t id = ids[(int64_t)t * id_stride + c];
            uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
            if (id >= 0 && id < ly.rows) {
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(ly.table + id * a.hd) + part);
                const float sc = __ldg(ly.scales + id * nblk + (part * 16) / a.blk);
                e4m3x4_scaled_to_bf16(v.x, sc, o0.x, o0.y);
                e4m3x4_scaled_to_bf16(v.y, sc, o0.z, o0.w);
                e4m3x4_scaled_to_bf16(v.z, sc, o1.x, o1.y);
                e4m3x4_scaled_to_bf16(v.w, sc, o1.z, o1.w);
            } else {
                set_err(a.err, ENGRAM_E_ROW);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(xs + (size_t)t * K + (size_t)c * a.hd) + 2 * part;
            dst[0] = o0;
            dst[1] = o1;
        }
    } else {
        for (int row = warp; row < n_ids; row += nwarps) {
            const int t = row / a.C, c = row % a.C;
            const int64_t id = ids[(int64_t)t * id_stride + c];
            const bool ok = id >= 0 && id < ly.rows;
            if (!ok && lane == 0) set_err(a.err, ENGRAM_E_ROW);
            q2k_row_to_smem(ly.table + (ok ? id : 0) * 84, ok, lane, xs + (size_t)t * K + (size_t)c * 256);
        }
    }
    __syncthreads();

    // ---- stream this CTA's wkv rows -------------------------------------------
    const uint4 *xs4 = reinterpret_cast<const uint4 *>(xs);
    for (; o < r1; o += nwarps) {
        const uint4 *wrow = reinterpret_cast<const uint4 *>(ly.wkv + (size_t)o * K);
        float acc[T];
#pragma unroll
        for (int t = 0; t < T; ++t) acc[t] = 0.0f;
        for (int base = 0; base < chunks; base += 32 * kGemvUnroll) {
            if (!prefetched) {
#pragma unroll
                for (int u = 0; u < kGemvUnroll; ++u) {
                    const int j = base + u * 32 + lane;
                    wv[u] = j < chunks ? ld_stream(wrow + j) : make_uint4(0, 0, 0, 0);
                }
            }
            prefetched = false;
#pragma unroll
            for (int u = 0; u < kGemvUnroll; ++u) {
                const int j = base + u * 32 + lane;
                if (j < chunks) {
#pragma unroll
                    for (int t = 0; t < T; ++t) acc[t] = dot8(wv[u], xs4[t * chunks + j], acc[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < T; ++t) {
            float v = acc[t];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
            acc[t] = v;
        }
        if (lane < T) {
            float v = acc[0];
#pragma unroll
            for (int t = 1; t < T; ++t) if (lane == t) v = acc[t];
            ly.kv[(size_t)lane * N + o] = (uint16_t)f32_to_bf16_bits(v);
        }
    }
}

size_t gemv_smem_bytes(int T, int K) { return (size_t)T * K * 2 + (size_t)kFusedHashMaxIds * 8; }

template <int T, bool HASH>
static cudaError_t launch_th(const GemvArgs &a, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t smem = (size_t)T * a.K * 2 + (HASH ? (size_t)T * a.C * 8 : 0);
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<T, HASH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_kernel<T, HASH>, kGemvThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int ctas_per_layer = (sms * per_sm) / a.L;
    const int max_useful = (a.N + 15) / 16;          // at least 16 rows a CTA
    if (ctas_per_layer > max_useful) ctas_per_layer = max_useful;
    if (ctas_per_layer < 1) ctas_per_layer = 1;
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
    switch (a.T) {
        case 0: return cudaSuccess;
        case 1: return launch_t<1>(a, s);
        case 2: return launch_t<2>(a, s);
        case 3: return launch_t<3>(a, s);
        case 4: return launch_t<4>(a, s);
        case 5: return launch_t<5>(a, s);
        case 6: return launch_t<6>(a, s);
        case 7: return launch_t<7>(a, s);
        case 8: return launch_t<8>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace engram
