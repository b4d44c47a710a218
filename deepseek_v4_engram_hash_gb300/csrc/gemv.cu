// gemv.cu -- the wkv projection for a few tokens (stage 3, 1 <= T <= 8), with
// the row gather and dequantisation (stage 2) fused into the x staging.
//
// kv[t, o] = bf16_rne(sum_i x[t, i] * wkv[o, i]), f32 accumulation
// (page "metrale_model_arch/deepseek_v41_ref/engram.rs", module doc, item 3).  At a few
// tokens the projection is a pass over wkv (251.7 MB a layer at V4.1 shape),
// so this kernel is shaped for HBM bandwidth, as the pages choose a GEMV over
// a tiled GEMM at m = 1 (page "spark_model/layers/attn_v41.rs", the doc of its
// kernel table: a bandwidth-bound GEMV in place of the tiled GEMM at one token).
//
// Grid: the layers' CTAs side by side, one an SM; the CTAs of a layer share
// its 16-row groups of wkv (handed out by a counter).  Prologue: the CTA
// hashes the step's ids for its layer and each MMA lane gathers its x
// fragments straight from the table rows (fp8 codes x scale, or Q2_K blocks)
// into registers -- the [T * C, head_dim] rows never touch HBM.  Main loop: a
// copy warp streams the groups' wkv rows into a shared-memory ring with bulk
// copies; 16 MMA warps multiply them by x on mma.sync m16n8k16 (bf16 in, f32
// accumulate) and hand their partial tiles to a reducing warp, which sums
// them and stores kv.  wkv may also be held as Q2_K
// blocks (page "spark_model/layers/engram_v41.rs", the doc of the layer weights:
// Q2_K wkv, 6x fewer bytes a token, byte-identical results): the
// same kernel then copies the blocks and decodes each lane's weights into its
// mma fragments, in the same order, so kv is bit-identical to the bf16 path on
// the dequantised weights.
#include "common.cuh"

namespace engram {

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
// bf16 wkv: the copy warp copies 16-row x 2048-wide pieces of the CTA's rows
// (4 KB contiguous a row) into a 3-stage ring, each stage completing an
// mbarrier by its byte count; the MMA warps read the pieces from shared memory
// and hand each stage back through a second mbarrier.  Larger copies keep
// more bytes in flight: 2 KB a row streamed one layer in 48.6 us, 3 KB in
// 39.4 us, 4 KB in 38.2 us.  Q2_K wkv: a stage is a
// whole 16-row group (16 x K/256 blocks of 84 bytes, contiguous in memory: one
// copy), six stages.  x is loop invariant for a warp (its k blocks are the
// same in every row group), so each lane gathers its x fragments once, straight
// from the table rows into registers; nothing but wkv goes through shared
// memory, and the ring's first stages are in flight before the dependency
// wait (two of three bf16 stages measured faster than all three).
//
// The dot product runs over k, so any permutation of k applied to both
// operands gives the same sum; lane (g = lane/4, q = lane%4) holds physical k
// 8q .. 8q+7 of each 32-wide k block: one 16-byte shared-memory read of rows
// g and g + 8 (bf16 ring rows padded by 64 bytes, so the 8 lanes of a phase
// hit distinct 16-byte bank groups) and token g's x feed two mma instructions.
// ---------------------------------------------------------------------------
constexpr int kMmaT = 8;
constexpr int kMmaWarps = 16;                           // MMA warps; then a copy warp and a reducing warp
constexpr int kMmaThreads = (kMmaWarps + 2) * 32;
constexpr int kMmaJ = 4;                                // 32-wide k blocks a warp per stage
constexpr int kStageKb = kMmaWarps * kMmaJ;             // 64 k blocks (2048 values) a bf16 stage
constexpr int kMmaSubMax = 3;                           // bf16 stages a 16-row group
static_assert(kMmaSubMax * kStageKb * 32 == kGemvMaxK, "x fragments cover K");
constexpr uint32_t kRowBytes = kStageKb * 64 + 64;      // one row's piece + bank padding
// Sleep hint of the reducing warp's waits, and of the copy warp's when the MMA
// warps are bound by the Q2_K decode (its waits are long; a sleeping warp
// leaves the issue slots to the decode: 53.9 -> 53.5 us a step).  Streaming
// bf16 wkv, the copy warp re-issues as soon as a stage frees: no sleep.
constexpr uint32_t kRoleSleepNs = 20000;
constexpr int kRedSlots = 2;                            // partial-tile slots between the MMA warps and the reducer
constexpr uint32_t kRedSlotFloats = kMmaWarps * 32 * 4; // one 16 x 8 f32 tile a warp
constexpr uint32_t kRedBytes = kRedSlots * kRedSlotFloats * 4;
static_assert((size_t)kFusedHashMaxIds * 8 <= kRedBytes, "hashed ids are staged in the partial buffer");

template <bool WQ2K>
struct Ring;
template <>
struct Ring<false> {
    static constexpr int kStages = 3;
    static constexpr int kPrefetch = 2;                                       // stages issued before the wait
    static constexpr uint32_t kStageBytes = 16 * kRowBytes;                   // 66 560
};
template <>
struct Ring<true> {
    static constexpr int kStages = 6;
    static constexpr int kPrefetch = 4;
    static constexpr uint32_t kStageBytes = 16 * (kGemvMaxK / 256) * 84;      // 32 256
};
template <bool WQ2K>
constexpr size_t ring_smem_bytes() {
    // ring, partial slots, the ring's full/empty and the slots' full/empty barriers, then the abort
    // and dependency flags, each ring slot's group and each partial slot's group
    return (size_t)Ring<WQ2K>::kStages * Ring<WQ2K>::kStageBytes + kRedBytes +
           (2 * Ring<WQ2K>::kStages + 2 * kRedSlots) * 8 + 16 + 4 * Ring<WQ2K>::kStages + 4 * kRedSlots;
}
static_assert(ring_smem_bytes<false>() <= 227 * 1024 && ring_smem_bytes<true>() <= 227 * 1024, "shared memory");

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

// Q2_K values in mma fragment form.  A 32-wide k block kk (0..7) of a 256-wide
// block is half = kk / 4, shift j = kk % 4; lane q's values 32 kk + 8q + e,
// e = 0..7, share the sub-block 8 half + 2j + q/2, and their quant bytes are
// qs[32 half + 8q + e] (block words 4 + 8 half + 2q and the next), the quant
// being (byte >> 2j) & 3.  A value is y = d*sc*q - dmin*m rounded once (d*sc*q
// and dmin*m are exact in f32, so fma(d*sc, q, -dmin*m) is that), then bf16:
// with one sub-block the lane's eight values take one of four, v[q].  v[0..3]
// are built once (q2k_table) and each pair (v[q_e], v[q_e+1]) is one byte
// permute of them, its selector nibbles 2q_e, 2q_e + 1, 2q_e+1, 2q_e+1 + 1: for
// four quants t, one a byte, t * 0x22 + 0x10101010 holds the selectors of
// pairs (0, 1) and, 16 bits up, (2, 3) (a permute reads the low 16 bits).
struct Q2kHalf {                  // what a lane needs of one half-block
    uint32_t q0, q1;              // its 8 quant bytes
    uint32_t sc01, sc23;          // the scale words of shifts 0,1 and 2,3
    float d, dmin;
};
__device__ __forceinline__ Q2kHalf q2k_half(const uint8_t *blk, int half, int q) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(blk);
    Q2kHalf h;
    h.q0 = w[4 + 8 * half + 2 * q];
    h.q1 = w[5 + 8 * half + 2 * q];
    h.sc01 = w[2 * half];
    h.sc23 = w[2 * half + 1];
    const __half2 dd = *reinterpret_cast<const __half2 *>(w + 20);
    h.d = __low2float(dd);
    h.dmin = __high2float(dd);
    return h;
}
// (d, -dmin/16) as an f32 pair (both exact)
__device__ __forceinline__ uint64_t q2k_dnm(const Q2kHalf &h) {
    return (uint64_t)__float_as_uint(h.d) | ((uint64_t)__float_as_uint(h.dmin * -0.0625f) << 32);
}
// The same table from the scale byte in place, in the main loop: sc & 15 and
// (sc & 0xF0) = 16 m both become exact floats by one OR each (2^23 + n, then
// one paired subtraction of 2^23), and one paired multiply by dnm = (d,
// -dmin/16) gives dl = d * sc and nml = -dmin * m -- both products exact in f32
// (11-bit d, dmin times at most 8 bits; -dmin/16 is exact), v[0] as fma(dl, 0,
// nml) for the sign of a zero -- so the values are bit-identical to
// q2k_table's.  Written as one asm block: the decode is bound by the integer
// pipe and the issue slots, and this form issued fewer instructions (one asm
// block: 45.4 against 46.3 us a step; the paired f32x2 steps: 42.9 against
// 43.8).
__device__ __forceinline__ uint2 q2k_table_b(uint32_t sc, uint64_t dnm) {
    uint2 r;
    asm("{\n\t.reg .b32 a, b;\n\t.reg .b64 ab, lm, k;\n\t.reg .f32 dl, nml, y0, y1, y2, y3;\n\t"
        "lop3.b32 a, %2, 0xF, 0x4B000000, 0xEA;\n\t"
        "lop3.b32 b, %2, 0xF0, 0x4B000000, 0xEA;\n\t"
        "mov.b64 ab, {a, b};\n\t"
        "mov.b64 k, 0x4B0000004B000000;\n\t"
        "sub.rn.f32x2 lm, ab, k;\n\t"
        "mul.rn.f32x2 lm, %3, lm;\n\t"
        "mov.b64 {dl, nml}, lm;\n\t"
        "fma.rn.f32 y0, dl, 0f00000000, nml;\n\t"
        "fma.rn.f32 y1, dl, 0f3F800000, nml;\n\t"
        "fma.rn.f32 y2, dl, 0f40000000, nml;\n\t"
        "fma.rn.f32 y3, dl, 0f40400000, nml;\n\t"
        "cvt.rn.bf16x2.f32 %0, y1, y0;\n\t"
        "cvt.rn.bf16x2.f32 %1, y3, y2;\n\t}"
        : "=r"(r.x), "=r"(r.y) : "r"(sc), "l"(dnm));
    return r;
}
// v[0..3] as bf16 pairs (v0 v1, v2 v3) for the sub-block scale byte sc
__device__ __forceinline__ uint2 q2k_table(uint32_t sc, float d, float dmin) {
    const float dl = __fmul_rn(d, small_u2f(sc & 15u));
    const float nml = -__fmul_rn(dmin, small_u2f(sc >> 4));
    return make_uint2(pack_bf16x2(__fmaf_rn(dl, 0.0f, nml), __fmaf_rn(dl, 1.0f, nml)),
                      pack_bf16x2(__fmaf_rn(dl, 2.0f, nml), __fmaf_rn(dl, 3.0f, nml)));
}
// Four values v[t_0..3] as bf16 pairs from quant word w (one value a byte, its
// quant at bits sh, sh + 1): t = (w >> sh) & 0x03030303, s = t * 0x22 +
// 0x10101010 holds the byte-permute selectors (nibbles 2t, 2t + 1) of values 0,
// 1 in its low half and of values 2, 3 in its high half.  Five integer-pipe
// instructions and one multiply-add per four weights, as one asm block: the
// same steps written in C++ issued about two more integer instructions per
// word (ncu: 20.0 M against 16.1 M a step; 51.7 against 46.3 us).  A 64-bit
// multiply-add giving both selectors at once measured slower (54.0 us), as did
// the high selector by a multiply-high (50.6 us).
__device__ __forceinline__ uint2 q2k_pick4_asm(uint2 v, uint32_t w, uint32_t sh) {
    uint2 r;
    asm("{\n\t.reg .b32 t, s, u;\n\t"
        "shr.b32 t, %2, %5;\n\t"
        "and.b32 t, t, 0x03030303;\n\t"
        "mad.lo.u32 s, t, 0x22, 0x10101010;\n\t"
        "shr.b32 u, s, 16;\n\t"
        "prmt.b32 %0, %3, %4, s;\n\t"
        "prmt.b32 %1, %3, %4, u;\n\t}"
        : "=r"(r.x), "=r"(r.y) : "r"(w), "r"(v.x), "r"(v.y), "r"(sh));
    return r;
}
// The same for quants already isolated in t (the one-time gather of x).
__device__ __forceinline__ uint2 q2k_pick4(uint2 v, uint32_t t) {
    const uint32_t s = t * 0x22u + 0x10101010u;
    return make_uint2(__byte_perm(v.x, v.y, s), __byte_perm(v.x, v.y, s >> 16));
}
__device__ __forceinline__ uint4 q2k_frag(const Q2kHalf &h, int j, int q) {
    // sub-block 8 half + 2j + q/2: byte 2 (j % 2) + q/2 of scale word j / 2
    const uint32_t sc = ((j < 2 ? h.sc01 : h.sc23) >> (8 * (2 * (j & 1) + (q >> 1)))) & 0xFFu;
    const uint2 v = q2k_table(sc, h.d, h.dmin);
    const uint2 a = q2k_pick4(v, (h.q0 >> (2 * j)) & 0x03030303u), b = q2k_pick4(v, (h.q1 >> (2 * j)) & 0x03030303u);
    return make_uint4(a.x, a.y, b.x, b.y);
}

// This lane's x fragments: token g, 32-wide k blocks kb = 64 s + 4w + (jj ^ q%2)
// of its warp w (jj = 0..3: lanes q and q ^ 1 take the blocks of a pair in
// opposite order, so that at Q2_K weights each builds one of the pair's two
// value tables and swaps it with the other), values x[g, 32 kb + 8q .. +7] as
// bf16 pairs -- from the plain x,
// or gathered from the layer's table rows ids[g * id_stride + c] (fp8 codes x
// their block's scale, or a Q2_K block) exactly as the row kernels dequantise
// them.  Ids first, then every load (an invalid id reads row 0 and gives
// zeros, raising ENGRAM_E_ROW), then the conversions: all of the lane's loads
// are in flight together.
__device__ __forceinline__ void gather_x(const GemvArgs &a, const GemvLayer &ly, const int64_t *ids,
                                         int64_t id_stride, int nsub, int warp, int g, int q,
                                         uint4 (&xr)[kMmaSubMax][kMmaJ]) {
    constexpr int NF = kMmaSubMax * kMmaJ;
    const int kblocks = a.K >> 5;
    const bool tok = g < a.T;
    const int t = tok ? g : 0;
    int k0[NF];
    bool need[NF];
#pragma unroll
    for (int f = 0; f < NF; ++f) {
        const int sub = f / kMmaJ, kb = sub * kStageKb + warp * kMmaJ + ((f % kMmaJ) ^ (q & 1));
        need[f] = tok && sub < nsub && kb < kblocks;
        k0[f] = (need[f] ? kb : 0) * 32 + 8 * q;
    }
    if (!a.gather) {
#pragma unroll
        for (int f = 0; f < NF; ++f) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(ly.x + (size_t)t * a.K + k0[f]));
            xr[f / kMmaJ][f % kMmaJ] = need[f] ? v : make_uint4(0, 0, 0, 0);
        }
        return;
    }
    // column c = k0 / head_dim, offset d0 = k0 % head_dim, scale block d0 / scale_block:
    // shifts when both are powers of two (every V4.1 shape), divisions otherwise
    int col[NF], d0[NF], sb[NF];
    if (((a.hd & (a.hd - 1)) | (a.blk & (a.blk - 1))) == 0) {
        const int hs = __ffs(a.hd) - 1, bs = __ffs(a.blk) - 1;
#pragma unroll
        for (int f = 0; f < NF; ++f) {
            col[f] = k0[f] >> hs;
            d0[f] = k0[f] & (a.hd - 1);
            sb[f] = d0[f] >> bs;
        }
    } else {
#pragma unroll
        for (int f = 0; f < NF; ++f) {
            col[f] = k0[f] / a.hd;
            d0[f] = k0[f] - col[f] * a.hd;
            sb[f] = d0[f] / a.blk;
        }
    }
    int64_t id[NF];
    bool ok[NF];
#pragma unroll
    for (int f = 0; f < NF; ++f) {
        const int64_t v = ids[(int64_t)t * id_stride + col[f]];
        ok[f] = need[f] && v >= 0 && v < ly.rows;
        id[f] = ok[f] ? v : 0;
        if (need[f] && !ok[f]) set_err(a.err, ENGRAM_E_ROW);
    }
    if (ly.fmt == ENGRAM_FMT_Q2K) {
        // head_dim 256: the warp's four k blocks of a stage are the four shifts of
        // half w % 2 of one block, so one row id and one half-block serve them
        Q2kHalf h[kMmaSubMax];
#pragma unroll
        for (int sub = 0; sub < kMmaSubMax; ++sub)
            h[sub] = q2k_half(ly.table + id[sub * kMmaJ] * 84, warp & 1, q);
#pragma unroll
        for (int f = 0; f < NF; ++f)
            xr[f / kMmaJ][f % kMmaJ] = ok[f] ? q2k_frag(h[f / kMmaJ], (f % kMmaJ) ^ (q & 1), q) : make_uint4(0, 0, 0, 0);
        return;
    }
    const int nblk = a.hd / a.blk;
    uint2 raw[NF];
    float sc[NF];
#pragma unroll
    for (int f = 0; f < NF; ++f)
        raw[f] = __ldg(reinterpret_cast<const uint2 *>(ly.table + id[f] * a.hd + d0[f]));
    if (ly.fmt == ENGRAM_FMT_FP8_E8M0) {
#pragma unroll
        for (int f = 0; f < NF; ++f)
            sc[f] = e8m0_to_f32(__ldg(static_cast<const uint8_t *>(ly.scales) + id[f] * nblk + sb[f]));
    } else {
#pragma unroll
        for (int f = 0; f < NF; ++f)
            sc[f] = __ldg(static_cast<const float *>(ly.scales) + id[f] * nblk + sb[f]);
    }
#pragma unroll
    for (int f = 0; f < NF; ++f) {
        uint4 o;
        e4m3x4_scaled_to_bf16(raw[f].x, sc[f], o.x, o.y);
        e4m3x4_scaled_to_bf16(raw[f].y, sc[f], o.z, o.w);
        xr[f / kMmaJ][f % kMmaJ] = ok[f] ? o : make_uint4(0, 0, 0, 0);
    }
}

// One CTA per SM.  The P CTAs that serve a layer take its 16-row groups from
// a counter (a.sched) in the order they ask, or else CTA c takes c, c + P,
// c + 2P, ...; either way the CTAs sweep the layer's wkv together (78.1
// against 78.9 us for contiguous runs of groups a CTA, both layers at one
// token; the counter 73.3 against 74.1 us a step).
// MMA warp w takes k blocks 64 s + 4w + j (s = 0 .. nsub-1, j = 0..3) of
// every row group -- for Q2_K weights the four shifts of half w % 2 of block
// 8 s + w / 2 -- lane q in the order j = 0 ^ q%2, 1 ^ q%2, 2 ^ q%2, 3 ^ q%2
// (K is a multiple of 64 on every path, so a warp's blocks in a stage are
// all valid, the first pair only, or none, alike for every lane; at Q2_K
// weights a warp with none multiplies zeros, which adds nothing), and the 16
// partial 16 x 8 tiles of a group are summed in warp order by the reducing
// warp; both weight formats follow this order exactly.  bf16: stage i is
// the CTA's group i / nsub, k blocks 64 (i % nsub) .. +63.  Q2_K: stage i is
// its group i.
template <bool HASH, bool WQ2K>
__global__ void __launch_bounds__(kMmaThreads, 1) gemv_mma_kernel(const __grid_constant__ GemvArgs a) {
    using R = Ring<WQ2K>;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int K = a.K, N = a.N, T = a.T;
    const uint32_t ring = smem_u32(smem_raw);
    float *red = reinterpret_cast<float *>(smem_raw + R::kStages * R::kStageBytes);
    int64_t *s_ids = reinterpret_cast<int64_t *>(red);                                   // until x is gathered
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw + R::kStages * R::kStageBytes + kRedBytes);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * R::kStages + 2 * kRedSlots);
    volatile int *dep_ok = abort_flag + 1;      // set once the kv stores may start (the dependency wait passed)
    volatile int *stage_grp = abort_flag + 4;   // [kStages]: the group of the stage in the slot, -1 at the end
    volatile int *slot_grp = stage_grp + R::kStages;   // [kRedSlots]: the group of the partials in the slot
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int b) { return bar0 + 8u * b; };
    auto empty = [&](int b) { return bar0 + 8u * (R::kStages + b); };
    auto red_full = [&](int b) { return bar0 + 8u * (2 * R::kStages + b); };
    auto red_empty = [&](int b) { return bar0 + 8u * (2 * R::kStages + kRedSlots + b); };

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
    const int spg = WQ2K ? 1 : nsub;                                     // stages a group
    const bool producer = warp == kMmaWarps;
    const bool reducer = warp == kMmaWarps + 1;

    if (threadIdx.x == 0) {
        for (int b = 0; b < R::kStages; ++b) {
            mbar_init(full(b), 1);
            mbar_init(empty(b), kMmaWarps);
        }
        for (int b = 0; b < kRedSlots; ++b) {
            mbar_init(red_full(b), kMmaWarps);
            mbar_init(red_empty(b), 1);
        }
        *abort_flag = 0;
        *dep_ok = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    const uint64_t pol = l2_evict_first();
    // The CTA's 16-row groups.  With a.sched, a per-layer counter hands them
    // out as the copy warps ask (CTAs whose copies land sooner take more: the
    // SMs of one launch stream at unequal rates, 11 us apart at the end of a
    // single-token step with a fixed share each); else cta, cta + P, cta + 2P, ...
    int issued = 0, cur = -1, grabs = 0;
    bool ended = false;
    auto next_group = [&]() {
        if (a.sched) return atomicAdd(a.sched + 2 * li, 1);
        return cta + (grabs++) * ctas_per_layer;
    };
    // Copy warp: stage `issued` into slot issued % kStages once the MMA warps
    // have released it, the slot's group written beside it.  Past the last
    // group the stage is an end marker (group -1, no bytes).  False once the
    // end marker is out or the CTA is aborting.
    auto issue_one = [&]() -> bool {
        const int i = issued, b = i % R::kStages;
        bool ok = true;
        if (lane == 0)
            ok = mbar_wait(empty(b), ((i / R::kStages) & 1) ^ 1, abort_flag, a.err, kWaitNs, WQ2K ? kRoleSleepNs : 0);
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
            ended = true;
            return false;
        }
        const int sub = WQ2K ? 0 : i % nsub;
        if (sub == 0) {
            int gnext = 0;
            if (lane == 0) gnext = next_group();
            cur = __shfl_sync(0xFFFFFFFFu, gnext, 0);
        }
        ++issued;
        if (cur >= groups_total) {
            if (lane == 0) {
                stage_grp[b] = -1;
                mbar_arrive(full(b));                  // completes the phase: no bytes
            }
            ended = true;
            return false;
        }
        if (lane == 0) stage_grp[b] = cur;             // published by the arrival below
        const uint32_t dst = ring + b * R::kStageBytes;
        if (WQ2K) {
            // the group's rows are contiguous: one copy of the 16-byte multiple,
            // the last 4..12 bytes (a short last group only) by plain stores
            const int r0 = cur * 16, nrows = min(16, N - r0);
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
            const int kb0 = sub * kStageKb;
            const uint32_t bytes = (uint32_t)min(kStageKb, kblocks - kb0) * 64u;
            const int r0 = cur * 16, nrows = min(16, N - r0);
            if (lane == 0) mbar_expect_tx(full(b), bytes * (uint32_t)nrows);
            __syncwarp();
            // row r0 + lane, columns kb0 * 32 ..: from the tiled copy (the group's
            // piece is one contiguous 64 KB tile) or from row-major wkv
            const uint16_t *src =
                ly.wkv_tiled ? ly.wkv_tiled + ((size_t)(cur * nsub + sub) * kTileRows + lane) * kTileCols
                             : ly.wkv + (size_t)(r0 + lane) * K + kb0 * 32;
            if (lane < nrows) bulk_load(dst + lane * kRowBytes, src, bytes, full(b), pol);
        }
        return true;
    };
    // the first stages need nothing computed: before the wait
    if (producer)
        for (int k = 0; k < R::kPrefetch && issue_one(); ++k) {
        }

    // Hashing here from a host position, the hash and the gather read only the
    // inputs, the constant tables and the cache entries of earlier steps; the
    // projection that wrote those had finished before the gate between it and
    // this grid let this grid launch (that gate signals its dependents only
    // after its own wait).  The wkv stream and the products read only
    // constants.  So all of that runs beside the previous step's gate, and only
    // the kv stores (which that gate reads) wait for it: the reducing warp
    // waits, and this grid signals its own dependents only after that wait.  A
    // device position is advanced by that gate (one step a launch): then
    // everything waits first -- unless the position stays put until this
    // step's own gate (the steps of a multi-step graph after the first).
    const bool early = HASH && (a.hash.start_pos_dev == nullptr || a.hash.pos_stable);
    if (a.pdl && !early) {
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

    if (producer) {
        while (!ended && issue_one()) {
        }
        // Let every copy already issued land before the CTA can leave.
        if (lane == 0)
            for (int d = 1; d <= R::kStages && issued - d >= 0; ++d) {
                const int i = issued - d;
                const uint64_t t0 = now_ns();
                while (!mbar_try(full(i % R::kStages), (i / R::kStages) & 1) && now_ns() - t0 < 10000000ull) {
                }
            }
        // The last of the layer's copy warps to finish resets its counters for
        // the next launch (launches of this kernel never overlap: the next one
        // starts after the gate that waits for this one).
        if (lane == 0 && a.sched) {
            __threadfence();
            if (atomicAdd(a.sched + 2 * li + 1, 1) == ctas_per_layer - 1) {
                atomicExch(a.sched + 2 * li, 0);
                atomicExch(a.sched + 2 * li + 1, 0);
            }
        }
        if (a.pdl && early && *dep_ok) griddep_launch();
        return;
    }

    if (reducer) {
        // Sums each group's 16 partial tiles in warp order and stores the group's
        // kv rows: lane l takes the four outputs of tile lane l (c0: row g,
        // token 2q; c1: row g, token 2q + 1; c2, c3: row g + 8), g = l / 4, q = l % 4.
        if (a.pdl && early) {
            griddep_wait();
            if (lane == 0) *dep_ok = 1;
            griddep_launch();
        }
        const int gg = lane >> 2, qq = lane & 3;
        for (int gi = 0;; ++gi) {
            const int slot = gi % kRedSlots;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(red_full(slot), (gi / kRedSlots) & 1, abort_flag, a.err, kWaitNs,
                                                   kRoleSleepNs)))
                break;
            const int grp = slot_grp[slot];
            if (grp < 0) break;
            const float4 *rb = reinterpret_cast<const float4 *>(red + slot * kRedSlotFloats);
            float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int w = 0; w < kMmaWarps; ++w) {
                const float4 p = rb[w * 32 + lane];
                v[0] += p.x;
                v[1] += p.y;
                v[2] += p.z;
                v[3] += p.w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(red_empty(slot));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = grp * 16 + gg + ((j & 2) ? 8 : 0), t = 2 * qq + (j & 1);
                if (r < N && t < T) ly.kv[(size_t)t * N + r] = (uint16_t)f32_to_bf16_bits(v[j]);
            }
        }
        return;
    }

    uint4 xr[kMmaSubMax][kMmaJ];
    gather_x(a, ly, ids, id_stride, nsub, warp, g, q, xr);
    mma_warps_sync();                      // every warp has read the hashed ids: the partial slots are free

    bool live = true;
    bool triggered = !(a.pdl && early);    // signalled already (or nothing to signal)
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
    // Q2_K: this lane's scale byte in a scale word, and the quant shifts 2j of blocks jj = 0, 1
    const int sc_byte = 8 * (warp & 1) + 2 * (q & 1) + (q >> 1);
    const uint32_t q_sh0 = 2u * (q & 1), q_sh1 = 2u - q_sh0;
    const int nblk_q = K >> 8;                                           // Q2_K blocks a row
    for (int gi = 0;; ++gi) {
        // the group's first stage names the group (-1: the end marker, the
        // same for every warp); a warp that finds the CTA aborting leaves
        const int i0 = gi * spg;
        const int grp = acquire(i0) ? stage_grp[i0 % R::kStages] : -1;
        if (!live) break;
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        if (grp >= 0) {
            if (WQ2K) {
                // this warp's blocks 8 s + w/2, half w % 2, of rows g and g + 8
                const uint8_t *row_lo = smem_raw + (gi % R::kStages) * R::kStageBytes + g * q2k_row;
                const uint8_t *row_hi = row_lo + 8 * q2k_row;
                // No test between the stages (their decode work then interleaves:
                // 43.8 against 45.2 us a step): a warp past the last block of a
                // narrower K decodes the row's last block instead, against x = 0
                // (its fragments are zero), adding exact zeros.
#pragma unroll
                for (int sub = 0; sub < kMmaSubMax; ++sub) {
                    const int blk = min(sub * 8 + (warp >> 1), nblk_q - 1);
                    const uint8_t *bl = row_lo + blk * 84, *bh = row_hi + blk * 84;
                    const Q2kHalf hl = q2k_half(bl, warp & 1, q);
                    const Q2kHalf hh = q2k_half(bh, warp & 1, q);
                    const uint64_t dl_ = q2k_dnm(hl), dh_ = q2k_dnm(hh);
                    // Block jj of the lane is shift j = jj ^ q%2.  At jj = 0, 2 the lane
                    // builds the value table of its sub-block (scale byte 2 (q%2) + q/2 of
                    // word jj/2); at jj = 1, 3 it needs shift j ^ 1 of the same pair,
                    // whose table lane q ^ 1 (same row, same sub-block) built at jj - 1.
                    uint2 vl[kMmaJ], vh[kMmaJ];
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        vl[2 * p] = q2k_table_b(bl[sc_byte + 4 * p], dl_);
                        vh[2 * p] = q2k_table_b(bh[sc_byte + 4 * p], dh_);
                    }
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        vl[2 * p + 1] = make_uint2(__shfl_xor_sync(0xFFFFFFFFu, vl[2 * p].x, 1),
                                                   __shfl_xor_sync(0xFFFFFFFFu, vl[2 * p].y, 1));
                        vh[2 * p + 1] = make_uint2(__shfl_xor_sync(0xFFFFFFFFu, vh[2 * p].x, 1),
                                                   __shfl_xor_sync(0xFFFFFFFFu, vh[2 * p].y, 1));
                    }
#pragma unroll
                    for (int jj = 0; jj < kMmaJ; ++jj) {
                        const uint32_t sh = ((jj & 1) ? q_sh1 : q_sh0) + ((jj & 2) ? 4u : 0u);    // 2j
                        const uint2 l0 = q2k_pick4_asm(vl[jj], hl.q0, sh);
                        const uint2 l1 = q2k_pick4_asm(vl[jj], hl.q1, sh);
                        const uint2 h0 = q2k_pick4_asm(vh[jj], hh.q0, sh);
                        const uint2 h1 = q2k_pick4_asm(vh[jj], hh.q1, sh);
                        const uint4 xb = xr[sub][jj];
                        mma_16816(c, l0.x, h0.x, l0.y, h0.y, xb.x, xb.y);
                        mma_16816(c, l1.x, h1.x, l1.y, h1.y, xb.z, xb.w);
                    }
                }
                release(gi);
            } else {
#pragma unroll
                for (int sub = 0; sub < kMmaSubMax; ++sub) {
                    if (sub < nsub) {
                        const int i = i0 + sub;
                        if (sub == 0 || acquire(i)) {
                            const uint32_t sa = ring + (i % R::kStages) * R::kStageBytes + a_off;
#pragma unroll
                            for (int jj = 0; jj < kMmaJ; ++jj) {
                                if (sub * kStageKb + warp * kMmaJ + jj < kblocks) {
                                    const uint32_t sj = sa + (uint32_t)((jj ^ (q & 1)) * 64);
                                    const uint4 lo = lds128(sj), hi = lds128(sj + 8 * kRowBytes);
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
            if (!live) break;
        }
        if (!triggered && *dep_ok) {
            griddep_launch();
            triggered = true;
        }
        // Hand the partial tile (or the end marker) to the reducing warp through
        // partial slot gi % kRedSlots, once the reducer has emptied its use gi - kRedSlots.
        const int slot = gi % kRedSlots;
        if (gi >= kRedSlots &&
            !__all_sync(0xFFFFFFFFu, mbar_wait(red_empty(slot), ((gi / kRedSlots) & 1) ^ 1, abort_flag, a.err)))
            break;
        if (grp >= 0)
            reinterpret_cast<float4 *>(red + slot * kRedSlotFloats)[warp * 32 + lane] = make_float4(c[0], c[1], c[2], c[3]);
        if (warp == 0 && lane == 0) slot_grp[slot] = grp;
        __syncwarp();
        if (lane == 0) mbar_arrive(red_full(slot));
        if (grp < 0) break;
    }
    if (!triggered && *dep_ok) griddep_launch();
}

template <bool HASH, bool WQ2K>
static cudaError_t launch_mma(const GemvArgs &a, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (a.T < 1 || a.T > kMmaT || a.K % (WQ2K ? 256 : 64) || a.K > kGemvMaxK || (WQ2K && a.K < 256))
        return cudaErrorInvalidValue;
    if (HASH && (size_t)a.T * a.C > (size_t)kFusedHashMaxIds) return cudaErrorInvalidValue;
    for (int l = 0; l < a.L; ++l) {
        const void *w = WQ2K ? static_cast<const void *>(a.layer[l].wkv_q2k) : static_cast<const void *>(a.layer[l].wkv);
        if (!w || reinterpret_cast<uintptr_t>(w) % 16) return cudaErrorInvalidValue;
    }
    const size_t smem = ring_smem_bytes<WQ2K>();
    static bool smem_set[64] = {};                   // per device, per instance
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!smem_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemv_mma_kernel<HASH, WQ2K>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        smem_set[dev] = true;
    }
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

static_assert(kStageKb * 32 == kTileCols && kTileRows == 16, "a bf16 ring stage is one tile of engram_tile_wkv");

// The engram_tile_wkv layout: one thread a 16-byte piece of the output, read
// from the row-major weights (K % 8 == 0), zero past the last row or column.
__global__ void __launch_bounds__(256) tile_wkv_kernel(const uint16_t *__restrict__ wkv, int N, int K,
                                                       uint16_t *__restrict__ tiled, int64_t pieces) {
    const int nchunks = (K + kTileCols - 1) / kTileCols;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < pieces;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int j8 = (int)(e % (kTileCols / 8));
        const int64_t row_of_tiles = e / (kTileCols / 8);       // (g * nchunks + c) * 16 + r
        const int r = (int)(row_of_tiles % kTileRows);
        const int64_t gc = row_of_tiles / kTileRows;
        const int c = (int)(gc % nchunks);
        const int64_t n = (gc / nchunks) * kTileRows + r;
        const int k = c * kTileCols + 8 * j8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (n < N && k < K) v = *reinterpret_cast<const uint4 *>(wkv + n * K + k);
        reinterpret_cast<uint4 *>(tiled)[e] = v;
    }
}

cudaError_t launch_tile_wkv(const uint16_t *wkv, int N, int K, uint16_t *tiled, cudaStream_t s) {
    const int64_t groups = (N + kTileRows - 1) / kTileRows, nchunks = (K + kTileCols - 1) / kTileCols;
    const int64_t pieces = groups * nchunks * kTileRows * (kTileCols / 8);
    if (pieces == 0) return cudaSuccess;
    const int64_t blocks = (pieces + 255) / 256;
    tile_wkv_kernel<<<(unsigned)(blocks < 152 * 32 ? blocks : 152 * 32), 256, 0, s>>>(wkv, N, K, tiled, pieces);
    return cudaGetLastError();
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
