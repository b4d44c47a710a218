// gemm_tc.cu -- the wkv projection on the 5th-generation tensor cores, one
// CTA a 128 x 256 tile (9..255 tokens; from 256 tokens the CTA-pair kernel of
// gemm_tc2.cu takes over, bit-identically).
//
// kv [M, N] = bf16_rne(x [M, K] . wkv [N, K]^T) with f32 accumulation
// (page "metrale_model_arch/deepseek_v41_ref/engram.rs", module doc, item 3), the dense
// contraction of the engram forward (2 x 4096 x 6144 x 20480 flop a layer at
// the V4.1 prefill shape).
//
// Persistent, warp-specialised, one CTA per SM, 6 warps:
//   warp 0      TMA producer: 128 x 64 tiles of x and 256 x 64 tiles of wkv
//               (128-byte swizzle) into a 4-stage shared-memory ring;
//   warp 1      owns the tensor memory (512 columns = two 128 x 256 f32
//               accumulators) and issues tcgen05.mma kind::f16 (M 128, N 256,
//               K 16) from one thread, committing each stage back to the
//               producer and each finished tile to the epilogue;
//   warps 2..5  epilogue: tcgen05.ld 32 columns at a time, bf16 round, store.
// The epilogue of tile i overlaps the main loop of tile i + 1.  Tiles are
// grouped (group_rows128 row tiles x all column tiles) so CTAs running
// together share x row blocks and wkv column blocks through L2.
//
// Every mbarrier wait is bounded (2 s on %globaltimer); on expiry the kernel
// sets ENGRAM_E_TIMEOUT, lets every role drain, frees its tensor memory and
// returns.
#include "tcgen05.cuh"

namespace engram {

namespace tc {

using namespace tcg;

constexpr int BM = 128, BN = 256, STAGES = 4;
constexpr int kThreads = 192;
constexpr uint32_t kStageA = BM * BK * 2;          // 16 KB
constexpr uint32_t kStageB = BN * BK * 2;          // 32 KB
constexpr uint32_t kStageBytes = kStageA + kStageB;
constexpr uint32_t kTmemCols = 512;                // two accumulators of BN columns
constexpr int kMaxL = kMaxLayers;
constexpr size_t kSmemBytes = 1024 + STAGES * kStageBytes + 256;

struct Params {
    CUtensorMap ta[kMaxL];
    CUtensorMap tb[kMaxL];
    uint16_t *kv[kMaxL];
    int L, M, N, K;
    int m_tiles, n_tiles, group_m;
    int *err;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

constexpr uint32_t kIdesc = idesc_bf16(BM, BN);

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(tmem_d), "l"(da), "l"(db), "r"(kIdesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;               // 1024-aligned for the swizzle
    uint8_t *gbase = smem_raw + (base - raw);
    // [stages: A | B] ... then barriers and bookkeeping
    uint8_t *aux = gbase + STAGES * kStageBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(aux);        // full[4] empty[4] tfull[2] tempty[2] drain
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(aux + 13 * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(aux + 13 * 8 + 4);
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    const uint32_t drain = bar0 + 8u * (2 * STAGES + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull(a), 1);
            mbar_init(tempty(a), 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32((const void *)tmem_slot)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int tiles_per_layer = p.m_tiles * p.n_tiles;
    const int n_tiles_total = tiles_per_layer * p.L;
    const int kblocks = p.K / BK;

    if (warp == 0) {
        if (lane == 0) {
            int it = 0;
            for (int tile = blockIdx.x; tile < n_tiles_total && !*abort_flag; tile += gridDim.x) {
                const int l = tile / tiles_per_layer, r = tile % tiles_per_layer;
                int mt, nt;
                tile_coords(r, p.m_tiles, p.n_tiles, p.group_m, mt, nt);
                const int m0 = mt * BM, n0 = nt * BN;
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (!mbar_wait(empty(s), ((it / STAGES) & 1) ^ 1, abort_flag, p.err)) break;
                    mbar_expect_tx(full(s), kStageBytes);
                    const uint32_t sa = base + s * kStageBytes;
                    tma_load_2d(sa, &p.ta[l], kb * BK, m0, full(s));
                    tma_load_2d(sa + kStageA, &p.tb[l], kb * BK, n0, full(s));
                }
            }
            // Let the copies already issued land before the CTA can leave.
            for (int s = 0; s < STAGES && it > 0; ++s) {
                const int last = it - 1 - s;
                if (last < 0) break;
                const uint64_t t0 = now_ns();
                while (!mbar_try(full(last % STAGES), (last / STAGES) & 1) && now_ns() - t0 < 10000000ull) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int it = 0, i = 0;
            for (int tile = blockIdx.x; tile < n_tiles_total && !*abort_flag; tile += gridDim.x, ++i) {
                const int acc = i & 1;
                if (!mbar_wait(tempty(acc), ((i >> 1) & 1) ^ 1, abort_flag, p.err)) break;
                tc_fence_after();
                const uint32_t d = tmem + acc * BN;
                bool ok = true;
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (!mbar_wait(full(s), (it / STAGES) & 1, abort_flag, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = base + s * kStageBytes;
                    const uint64_t da = sdesc(sa), db = sdesc(sa + kStageA);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)                 // +32 bytes = 2 in the address field
                        mma_bf16(d, da + 2u * k, db + 2u * k, (kb | k) != 0);
                    mma_commit(empty(s));
                }
                if (!ok) break;
                mma_commit(tfull(acc));
            }
            // Drain: every MMA issued so far has finished before TMEM is freed.
            mma_commit(drain);
            const uint64_t t0 = now_ns();
            while (!mbar_try(drain, 0) && now_ns() - t0 < 100000000ull) {
            }
        }
        __syncwarp();
    } else {
        // Epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31, one row each.
        const int q = warp & 3;
        const int row = 32 * q + lane;
        int i = 0;
        for (int tile = blockIdx.x; tile < n_tiles_total; tile += gridDim.x, ++i) {
            const int acc = i & 1;
            const bool ok = mbar_wait(tfull(acc), (i >> 1) & 1, abort_flag, p.err);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;          // reconverge before .sync.aligned loads
            tc_fence_after();
            const int l = tile / tiles_per_layer, r = tile % tiles_per_layer;
            int mt, nt;
            tile_coords(r, p.m_tiles, p.n_tiles, p.group_m, mt, nt);
            const int m = mt * BM + row, n0 = nt * BN;
            uint16_t *out = p.kv[l] + (size_t)m * p.N;
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + acc * BN + c, v);
                if (m < p.M) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int n = n0 + c + 8 * j;
                        if (n < p.N) {
                            uint4 o;
                            o.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1]));
                            o.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3]));
                            o.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5]));
                            o.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]));
                            *reinterpret_cast<uint4 *>(out + n) = o;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty(acc));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

}  // namespace tc

namespace tcg {

// ---------------------------------------------------------------------------
// Host side: tensor maps through the driver entry point (no -lcuda link).
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool make_map(CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool have_tensor_maps() { return encode_fn() != nullptr; }

}  // namespace tcg

bool gemm_tc_supported(int M, int N, int K) {
    return M >= 1 && K >= tcg::BK && K % tcg::BK == 0 && N % 8 == 0 && N >= 8 && tcg::have_tensor_maps();
}

// L layers: x[l] [M, K] and wkv[l] [N, K] -> kv[l] [M, N], one persistent launch.
cudaError_t launch_gemm_tc(int L, const uint16_t *const *x, const uint16_t *const *wkv, uint16_t *const *kv,
                           int M, int N, int K, int *err, cudaStream_t s, bool pdl, const GemmTail *tail) {
    using namespace tc;
    if (L < 1 || L > kMaxL) return cudaErrorInvalidValue;
    // 256 tokens and up: 256 x 256 tiles on CTA pairs (gemm_tc2.cu), bit-identical
    // except for tiles of a last wave cut along K (only with `tail`)
    if (M >= 256) return launch_gemm_tc2(L, x, wkv, kv, M, N, K, err, s, pdl, tail);
    Params p{};
    for (int l = 0; l < L; ++l) {
        if (!make_map(&p.ta[l], x[l], (uint64_t)K, (uint64_t)M, BM)) return cudaErrorInvalidValue;
        if (!make_map(&p.tb[l], wkv[l], (uint64_t)K, (uint64_t)N, BN)) return cudaErrorInvalidValue;
        p.kv[l] = kv[l];
    }
    p.L = L;
    p.M = M;
    p.N = N;
    p.K = K;
    p.m_tiles = (M + BM - 1) / BM;
    p.n_tiles = (N + BN - 1) / BN;
    p.group_m = group_rows128(p.m_tiles);
    p.err = err;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    static bool attr[64] = {};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr[dev] = true;
    }
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int tiles = p.m_tiles * p.n_tiles * L;
    const int grid = tiles < sms ? tiles : sms;
    gemm_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace engram
