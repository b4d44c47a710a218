// gemm_tc2.cu -- the prefill wkv projection on CTA pairs (tcgen05 cta_group::2).
//
// kv [M, N] = bf16_rne(x [M, K] . wkv [N, K]^T) with f32 accumulation
// (page "metrale_model_arch/deepseek_v41_ref/engram.rs", module doc, item 3), as in
// gemm_tc.cu, but a cluster of two CTAs computes one 256 x 256 tile: CTA r of
// the pair holds x rows m0 + 128 r .. +127 and wkv rows n0 + 128 r .. +127 of
// every 64-wide k step in its own shared memory, and one thread of CTA 0
// issues tcgen05.mma.cta_group::2 (M 256, N 256, K 16), which reads both
// CTAs' halves and accumulates each CTA's 128 rows x 256 columns in that CTA's
// tensor memory.  A CTA stages 32 KB a k step for the same 4.2 MFLOP a CTA
// that gemm_tc.cu stages 48 KB for, so seven stages fit where four did
// (seven against six: 1012 against 1017 us at 4096 tokens, 165 against 167 us
// at 512).
//
// Roles (6 warps a CTA):
//   warp 0      TMA producer of this CTA's halves; the copies of both CTAs
//               complete their bytes on CTA 0's "full" barrier (cta_group::2
//               copies), whose expected count CTA 0's producer sets;
//   warp 1      CTA 0: owns the MMA; waits on its full barrier, commits each
//               stage back to both CTAs' "empty" barriers and each finished
//               tile to both CTAs' "tfull" barriers.  CTA 1: idle;
//   warps 2..5  epilogue of this CTA's 128 rows; CTA 0's "tempty" barrier
//               counts the epilogue warps of both CTAs.
// Every mbarrier wait is bounded (2 s); on expiry the kernel raises
// ENGRAM_E_TIMEOUT, every role of both CTAs runs out its loops, and both CTAs
// meet at the final cluster barrier before the tensor memory is freed.
#include "tcgen05.cuh"

namespace engram {

namespace tc2 {

using namespace tcg;

constexpr int BMC = 128;                            // rows a CTA (M 256 a pair)
constexpr int BN = 256, STAGES = 7;            // 7 x 32 KB ring: 230.7 KB of shared memory
constexpr int kThreads = 192;
constexpr uint32_t kStageA = BMC * BK * 2;          // 16 KB
constexpr uint32_t kStageB = (BN / 2) * BK * 2;     // 16 KB: this CTA's half of the wkv tile
constexpr uint32_t kStageBytes = kStageA + kStageB;
constexpr int kAcc = 2;                             // accumulators in tensor memory (512 columns)
constexpr uint32_t kTmemCols = kAcc * BN;
constexpr int kMaxL = kMaxLayers;
constexpr size_t kSmemBytes = 1024 + STAGES * kStageBytes + 256;

struct Params {
    CUtensorMap ta[kMaxL];
    CUtensorMap tb[kMaxL];
    CUtensorMap tbs[kMaxL];                         // wkv boxes of BN / (2 split) rows (tail sub-tiles)
    uint16_t *kv[kMaxL];
    int L, M, N, K;
    int m_tiles, n_tiles, group_m;                  // m_tiles: 256-row pair tiles
    int full_per_pair;                              // whole tiles every pair takes first
    int tail_tiles, split;                          // the last tiles, each cut into `split` column parts
    int ksplit, kb_per;                             // or (ksplit > 1) into ksplit K ranges of kb_per k steps
    float *part;                                    // K-split partials [tail tile][ksplit][256 columns][256 rows]
    int n_pairs;                                    // CTA pairs of the launch
    int pdl;                                        // wait for the previous kernel after the set-up
    int *err;
};

// Work item k of a pair: its whole tiles first (tile pair + k P, P pairs),
// then the last tail_tiles tiles spread over every pair, either as column
// parts u = pair + j P (split parts of BN / split columns each: a part keeps
// every output's K order, so results do not depend on it) or, with ksplit > 1,
// as K ranges: item u = pair is range u % ksplit of tail tile u / ksplit (at
// most one an item a pair, since tail_tiles * ksplit <= P).  A K range's
// product goes to an f32 partial tile; gemm_tail_fixup_kernel, launched next,
// adds each tile's ranges in range order and stores its bf16 kv.
struct Work {
    int l, mt, nt, n0, width;                      // n0: first column of the item
    int kb0, kb1;                                  // the item's k steps
    int tail, j;                                   // K-split item: tail tile and range (tail < 0 otherwise)
};
__device__ __forceinline__ bool work_item(const Params &p, int pair, int n_pairs, int k, Work &w) {
    const int tiles_per_layer = p.m_tiles * p.n_tiles;
    int tile, part = 0;
    w.width = BN;
    w.kb0 = 0;
    w.kb1 = p.K / BK;
    w.tail = -1;
    w.j = 0;
    if (k < p.full_per_pair) {
        tile = pair + k * n_pairs;
        if (tile >= tiles_per_layer * p.L) return false;
    } else if (p.ksplit > 1) {
        const int u = pair + (k - p.full_per_pair) * n_pairs;
        if (u >= p.tail_tiles * p.ksplit) return false;
        w.tail = u / p.ksplit;
        w.j = u % p.ksplit;
        tile = p.full_per_pair * n_pairs + w.tail;
        w.kb0 = w.j * p.kb_per;
        w.kb1 = min(w.kb1, w.kb0 + p.kb_per);
    } else {
        const int u = pair + (k - p.full_per_pair) * n_pairs;
        if (u >= p.tail_tiles * p.split) return false;
        tile = p.full_per_pair * n_pairs + u / p.split;
        part = u % p.split;
        w.width = BN / p.split;
    }
    w.l = tile / tiles_per_layer;
    tile_coords(tile % tiles_per_layer, p.m_tiles, p.n_tiles, p.group_m, w.mt, w.nt);
    w.n0 = w.nt * BN + part * w.width;
    return true;
}

// 2D tile load into this CTA's shared memory whose bytes complete on an
// mbarrier of either CTA of the pair (`bar`: a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int x, int y,
                                                 uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// The shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on an mbarrier of either CTA of the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// M 256 for the pair, N = the item's width (256, or a tail part's 128 / 64).
__device__ __forceinline__ void mma_pair(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(tmem_d), "l"(da), "l"(db), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the mbarrier at this offset in both CTAs of the pair when
// every MMA issued so far has completed.
__device__ __forceinline__ void commit_both(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        ::"r"(bar), "h"((uint16_t)0x3)
        : "memory");
}
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_tc2_kernel(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;       // the same offset in both CTAs
    uint8_t *aux = smem_raw + (base - raw) + STAGES * kStageBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(aux);  // full[S] empty[S] tfull[2] tempty[2] drain
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(aux + (2 * STAGES + 5) * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(aux + (2 * STAGES + 5) * 8 + 4);
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    const uint32_t drain = bar0 + 8u * (2 * STAGES + 4);

    const uint32_t rank = cluster_rank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);                      // CTA 0's: its producer; bytes of both CTAs
            mbar_init(empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull(a), 1);
            mbar_init(tempty(a), 8);                    // four epilogue warps in each CTA
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32((const void *)tmem_slot)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();                                     // both CTAs' barriers exist before any remote arrival
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched early (programmatic dependent of the row gather): the set-up
    // above ran beside the gather's last CTAs; x is read only after this.
    // (The gate after the GEMM stays a plain launch: launched early, its CTAs
    // beside the GEMM's made the 512-token step 2 % slower.)
    if (p.pdl) griddep_wait();

    const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
    Work w;

    if (warp == 0) {
        if (lane == 0) {
            int it = 0;
            for (int k = 0; work_item(p, pair, n_pairs, k, w) && !*abort_flag; ++k) {
                const int half = w.width / 2;                 // wkv rows this CTA stages
                const int m0 = w.mt * 2 * BMC + (int)rank * BMC, n0 = w.n0 + (int)rank * half;
                const CUtensorMap *mb = w.width == BN ? &p.tb[w.l] : &p.tbs[w.l];
                const uint32_t bytes = kStageA + (uint32_t)half * BK * 2;
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (!mbar_wait(empty(s), ((it / STAGES) & 1) ^ 1, abort_flag, p.err)) break;
                    if (rank == 0) mbar_expect_tx(full(s), 2 * bytes);
                    const uint32_t sa = base + s * kStageBytes, fb = mapa(full(s), 0);
                    tma_load_2d_pair(sa, &p.ta[w.l], kb * BK, m0, fb);
                    tma_load_2d_pair(sa + kStageA, mb, kb * BK, n0, fb);
                }
            }
            // Let the copies already issued land before the pair can leave (CTA 0's
            // full barriers count the bytes of both CTAs).
            for (int d = 1; rank == 0 && d <= STAGES && it - d >= 0; ++d) {
                const int last = it - d;
                const uint64_t t0 = now_ns();
                while (!mbar_try(full(last % STAGES), (last / STAGES) & 1) && now_ns() - t0 < 10000000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            int it = 0, i = 0;
            for (int k = 0; work_item(p, pair, n_pairs, k, w) && !*abort_flag; ++k, ++i) {
                const int acc = i % kAcc;
                if (!mbar_wait(tempty(acc), ((i / kAcc) & 1) ^ 1, abort_flag, p.err)) break;
                tc_fence_after();
                const uint32_t d = tmem + acc * BN;
                const uint32_t idesc = idesc_bf16(2 * BMC, w.width);
                bool ok = true;
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (!mbar_wait(full(s), (it / STAGES) & 1, abort_flag, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = base + s * kStageBytes;
                    const uint64_t da = sdesc(sa), db = sdesc(sa + kStageA);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)              // +32 bytes = 2 in the address field
                        mma_pair(d, da + 2u * kk, db + 2u * kk, idesc, (kb != w.kb0) | (kk != 0));
                    commit_both(empty(s));
                }
                if (!ok) break;
                commit_both(tfull(acc));
            }
            // Drain: every MMA issued so far has finished before the pair can free tensor memory.
            commit_both(drain);
            const uint64_t t0 = now_ns();
            while (!mbar_try(drain, 0) && now_ns() - t0 < 100000000ull) {
            }
        }
        __syncwarp();
    } else {
        // Epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 -- rows of this CTA's half.
        const int q = warp & 3;
        const int row = (int)rank * BMC + 32 * q + lane;
        int i = 0;
        for (int k = 0; work_item(p, pair, n_pairs, k, w); ++k, ++i) {
            const int acc = i % kAcc;
            const bool ok = mbar_wait(tfull(acc), (i / kAcc) & 1, abort_flag, p.err);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;          // reconverge before .sync.aligned loads
            tc_fence_after();
            const int m = w.mt * 2 * BMC + row, n0 = w.n0;
            uint16_t *out = p.kv[w.l] + (size_t)m * p.N;
            if (w.tail >= 0) {
                // K-split item: this CTA's 128 rows of the f32 partial, column-major
                // ([column][row]: a warp's 32 rows of one column are one 128-byte
                // line); gemm_tail_fixup_kernel adds the ranges after the launch
                float *pcol = p.part + (size_t)(w.tail * p.ksplit + w.j) * BN * (2 * BMC) + row;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t v[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + acc * BN + c, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) pcol[(size_t)(c + j) * (2 * BMC)] = __uint_as_float(v[j]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa(tempty(acc), 0));
                continue;
            }
#pragma unroll 1
            for (int c = 0; c < w.width; c += 32) {
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
            if (lane == 0) mbar_arrive_cluster(mapa(tempty(acc), 0));
        }
    }

    // Both CTAs meet here: no remote arrival, copy or MMA of either is still in flight.
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// The K-split tiles of the last wave: kv = bf16(sum of the ksplit partials in
// range order) -- a fixed order, so the result does not depend on timing.  A
// thread takes 8 columns of one row; the 32 threads of a warp take 32
// consecutive rows, so every partial load is a 128-byte line.
__global__ void __launch_bounds__(256) gemm_tail_fixup_kernel(const __grid_constant__ Params p) {
    const int tpt = BN / 8 * (2 * BMC);                              // threads a tail tile
    const int gid = blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= p.tail_tiles * tpt) return;
    const int tail = gid / tpt, r = gid % tpt;
    const int row = r % (2 * BMC), c0 = (r / (2 * BMC)) * 8;
    const int tile = p.full_per_pair * p.n_pairs + tail;
    const int tiles_per_layer = p.m_tiles * p.n_tiles;
    const int l = tile / tiles_per_layer;
    int mt, nt;
    tile_coords(tile % tiles_per_layer, p.m_tiles, p.n_tiles, p.group_m, mt, nt);
    const int m = mt * 2 * BMC + row, n = nt * BN + c0;
    if (m >= p.M || n >= p.N) return;
    const float *src = p.part + (size_t)tail * p.ksplit * BN * (2 * BMC) + (size_t)c0 * (2 * BMC) + row;
    float a[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) a[e] = __ldcg(src + e * (2 * BMC));
    for (int j = 1; j < p.ksplit; ++j) {
        const float *pj = src + (size_t)j * BN * (2 * BMC);
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] += __ldcg(pj + e * (2 * BMC));
    }
    *reinterpret_cast<uint4 *>(p.kv[l] + (size_t)m * p.N + n) =
        make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                   pack_bf16x2(a[6], a[7]));
}

}  // namespace tc2

// L layers: x[l] [M, K] and wkv[l] [N, K] -> kv[l] [M, N], one persistent
// launch of CTA pairs.
cudaError_t launch_gemm_tc2(int L, const uint16_t *const *x, const uint16_t *const *wkv, uint16_t *const *kv,
                            int M, int N, int K, int *err, cudaStream_t s, bool pdl, const GemmTail *tail) {
    using namespace tc2;
    if (L < 1 || L > kMaxL || M < 1 || K < BK || K % BK || N < 8 || N % 8) return cudaErrorInvalidValue;
    Params p{};
    for (int l = 0; l < L; ++l) {
        if (!make_map(&p.ta[l], x[l], (uint64_t)K, (uint64_t)M, BMC)) return cudaErrorInvalidValue;
        if (!make_map(&p.tb[l], wkv[l], (uint64_t)K, (uint64_t)N, BN / 2)) return cudaErrorInvalidValue;
        p.kv[l] = kv[l];
    }
    p.L = L;
    p.M = M;
    p.N = N;
    p.K = K;
    p.m_tiles = (M + 2 * BMC - 1) / (2 * BMC);
    p.n_tiles = (N + BN - 1) / BN;
    p.group_m = group_rows128(2 * p.m_tiles) / 2 > 0 ? group_rows128(2 * p.m_tiles) / 2 : 1;   // in pair tiles
    p.err = err;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    static bool attr[64] = {};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr[dev] = true;
    }
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int tiles = p.m_tiles * p.n_tiles * L;
    const int pairs = tiles < sms / 2 ? tiles : sms / 2;
    // The partial last wave: its R tiles cut into `split` column parts (2 or 4)
    // when that shortens it.  A part still stages the whole 16 KB x tile every k
    // step, so it is bound by staging, not by its MMA: a half part costs about
    // 6/8 of a whole tile, a quarter part 5/8 (measured: quarter parts made the
    // 4096-token GEMM's 52-tile tail slower, the 512-token one's faster).
    const int R = tiles % pairs;
    // With partial-tile scratch, a last wave of at most half the pairs is cut
    // along K instead: each of its R tiles into ksplit ranges (ksplit <= 8, so
    // the fix-up reads at most eight partials), one range a pair; the wave then
    // costs about 1 / ksplit of a round plus the fix-up.
    const int kblocks = K / BK;
    if (tail && tail->part && R > 0 && 2 * R <= pairs && R <= kTailItems) {
        int ks = pairs / R;
        ks = ks > 8 ? 8 : ks;
        ks = ks > kblocks ? kblocks : ks;
        const int kb_per = (kblocks + ks - 1) / ks;
        p.ksplit = (kblocks + kb_per - 1) / kb_per;              // no empty range
        p.kb_per = kb_per;
        p.part = tail->part;
        p.split = 1;
        p.full_per_pair = (tiles - R) / pairs;
        p.tail_tiles = R;
    }
    int split = 1, best = R > 0 && p.ksplit < 2 ? 8 : 0;
    for (int c = 2; c <= 4 && R > 0; c *= 2) {
        const int cost = ((R * c + pairs - 1) / pairs) * (c == 2 ? 6 : 5);
        if (cost < best) {
            best = cost;
            split = c;
        }
    }
    if (p.ksplit >= 2) {
        // set above
    } else if ((p.split = split) > 1) {
        p.full_per_pair = (tiles - R) / pairs;
        p.tail_tiles = R;
        for (int l = 0; l < L; ++l)
            if (!make_map(&p.tbs[l], wkv[l], (uint64_t)K, (uint64_t)N, (uint32_t)(BN / (2 * split))))
                return cudaErrorInvalidValue;
    } else {
        p.full_per_pair = (tiles + pairs - 1) / pairs;
        p.tail_tiles = 0;
    }
    p.pdl = pdl ? 1 : 0;
    p.n_pairs = pairs;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_tc2_kernel, p);
    if (e != cudaSuccess || p.ksplit < 2) return e;
    const int threads = p.tail_tiles * (BN / 8) * (2 * BMC);
    gemm_tail_fixup_kernel<<<(threads + 255) / 256, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace engram
