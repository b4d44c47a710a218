// common.cuh -- device helpers and launcher declarations shared by the
// libengram translation units (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/engram.h"

namespace engram {

constexpr int kMaxLayers = 4;
constexpr int kMaxNgram = 16;
constexpr int kSmallT = 8;          // tokens at or below this run the fused GEMV

// ---------------------------------------------------------------------------
// Sticky device error word: the first error code wins; kernels never trap.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_err(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Round-to-nearest-even f32 -> bf16 bits (cvt.rn.bf16.f32).
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float x) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Four e4m3 codes (one 32-bit word, little-endian) times a power-of-two
// scale -> four bf16, packed in two words.  e4m3 -> f16 is exact (hardware
// cvt), f16 -> f32 exact, the f32 multiply by 2^k is exact unless it leaves
// the f32 range, and the final cvt.rn.bf16 is round-to-nearest-even: the
// same value as bf16_rne(e4m3_to_f32(b) * scale) in the CPU reference.
__device__ __forceinline__ void e4m3x4_scaled_to_bf16(uint32_t codes, float scale,
                                                      uint32_t &out01, uint32_t &out23) {
    __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(codes & 0xFFFFu), __NV_E4M3);
    __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(codes >> 16), __NV_E4M3);
    float2 a = __half22float2(*reinterpret_cast<__half2 *>(&lo));
    float2 b = __half22float2(*reinterpret_cast<__half2 *>(&hi));
    out01 = pack_bf16x2(__fmul_rn(a.x, scale), __fmul_rn(a.y, scale));
    out23 = pack_bf16x2(__fmul_rn(b.x, scale), __fmul_rn(b.y, scale));
}

// e8m0 byte -> f32 scale 2^(code - 127): the byte is the biased exponent
// (code 0 is the subnormal 2^-127, code 255 NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t code) {
    return __uint_as_float(code == 0u ? 0x00400000u : (code == 255u ? 0x7FC00000u : code << 23));
}

// The scale of fp8 row `id`, block `b`: f32 (fmt FP8) or an e8m0 byte (FP8_E8M0).
__device__ __forceinline__ float fp8_row_scale(const void *scales, int fmt, int64_t idx) {
    return fmt == ENGRAM_FMT_FP8_E8M0 ? e8m0_to_f32(__ldg(static_cast<const uint8_t *>(scales) + idx))
                                      : __ldg(static_cast<const float *>(scales) + idx);
}

// One Q2_K value: d * (sc & 15) * q - dmin * (sc >> 4); every product is exact
// in f32, so only the subtraction rounds.
__device__ __forceinline__ float q2k_value(float d, float dmin, uint32_t sc, uint32_t q) {
    return __fsub_rn(__fmul_rn(__fmul_rn(d, (float)(sc & 15u)), (float)q),
                     __fmul_rn(dmin, (float)(sc >> 4)));
}

// One lane's share of a Q2_K block decode: the warp holds the block's 21
// little-endian words in lanes 0..20 (`word`); lane l returns the bf16 values
// 8l .. 8l+7 packed in a uint4.  For v = 8l + e: half = l/16, j = (l%16)/4,
// the quant bytes are qs[32 half + 8 (l%4) + e] (block words 4 + 8 half +
// 2 (l%4) and the next), the sub-block is 8 half + 2j + (l%4)/2, and the
// quant is (byte >> 2j) & 3.  All 32 lanes must call it (shuffles).
__device__ __forceinline__ uint4 q2k_lane_decode(uint32_t word, int lane) {
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
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t byte = ((e < 4 ? q0 : q1) >> (8 * (e & 3))) & 0xFFu;
        y[e] = q2k_value(d, dmin, sc, (byte >> (2 * j)) & 3u);
    }
    return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                      pack_bf16x2(y[6], y[7]));
}

// ---------------------------------------------------------------------------
// Launchers (host side, defined in the kernel translation units)
// ---------------------------------------------------------------------------
struct HashArgs {
    const int32_t *ids;
    int32_t B, T;
    int64_t start_pos;              // the start position, or (with start_pos_dev) an offset added to it
    const int64_t *start_pos_dev;   // when set, the start position is read here (device memory)
    int32_t pos_stable;             // the device position is not written before this step's own gate
    const int64_t *token_map;
    int64_t vocab, pad_id;
    const int64_t *mult, *primes, *offsets;
    const uint64_t *bm;       // per prime: floor(2^64 / p) (0 for p = 1)
    const uint64_t *wrap;     // per prime: 2^64 mod p
    int32_t L, ng, H;
    int64_t *cache;
    int64_t max_seq;
    int64_t *out;
    int *err;
};
cudaError_t launch_hash(const HashArgs &a, cudaStream_t s);

// The call's start position: the host value, or the device-resident one plus
// the host offset (steps after the first of a multi-step graph).
// A device position that does not fit the cache raises ENGRAM_E_CAPACITY;
// the caller then skips every cache access (false).
__device__ __forceinline__ bool hash_start(const HashArgs &a, int64_t &sp) {
    sp = a.start_pos_dev ? *a.start_pos_dev + a.start_pos : a.start_pos;
    if (sp < 0 || sp + a.T > a.max_seq) {
        set_err(a.err, ENGRAM_E_CAPACITY);
        return false;
    }
    return true;
}

// Compressed id of input token s of sequence b (the token_map lookup); an id
// outside token_map raises ENGRAM_E_TOKEN and reads as unmapped (-1).
__device__ __forceinline__ int64_t hash_compress(const HashArgs &a, int b, int64_t s) {
    const int32_t id = a.ids[(int64_t)b * a.T + s];
    if (id < 0 || (int64_t)id >= a.vocab) {
        set_err(a.err, ENGRAM_E_TOKEN);
        return -1;
    }
    return a.token_map[id];
}

// rem_euclid(x, p) for the i64 value whose bits are `u` and 0 < p < 2^63, by
// Barrett reduction (no 64-bit division): with m = floor(2^64 / p),
// q = floor(u m / 2^64) is floor(u / p) or one less, so u - q p lies in
// [0, 2p) and one subtraction finishes u mod p.  A negative x is u - 2^64,
// so its remainder is (u mod p) - (2^64 mod p), lifted into [0, p).
__device__ __forceinline__ uint64_t rem_euclid_barrett(uint64_t u, uint64_t p, uint64_t m, uint64_t wrap) {
    if (p == 1) return 0;
    const uint64_t q = __umul64hi(u, m);
    uint64_t r = u - q * p;
    if (r >= p) r -= p;
    if ((int64_t)u < 0) r = r >= wrap ? r - wrap : r + p - wrap;
    return r;
}

// Row id of (sequence b, position start_pos + s, layer li, column col):
// the hash of page "metrale_model_arch/deepseek_v41_ref/engram.rs" (module doc,
// item 1) and page "spark_model/layers/engram_v41.rs" (module doc, item 1):
//   w_j = cache[p - j] while no shift up to j reaches before position 0 or an
//         unmapped (-1) id, else pad_id;
//   X_n = XOR_{j=0..n} (w_j *wrap m_j)  for the (n+1)-gram, n = col / H + 1;
//   id  = rem_euclid(X_n, prime[col]) + offset[col],
// all i64 with wrap; X_n is formed slot by slot as the window is read, and
// the remainder is taken by Barrett reduction (rem_euclid_barrett).  Ids
// of this call come from the input through token_map, older positions from
// the cache, so no thread depends on another thread's cache write.
__device__ __forceinline__ int64_t hash_one(const HashArgs &a, int64_t sp, int b, int s, int li, int col) {
    const int C = (a.ng - 1) * a.H;
    const int64_t pos = sp + s;
    const int n_top = col / a.H + 1;
    const int64_t *m = a.mult + (int64_t)li * a.ng;
    // the window's token at each shift, folded into the rolling XOR as it is formed
    uint64_t rolling = 0;
    bool blocked = false;
    for (int shift = 0; shift <= n_top; ++shift) {
        int64_t src;
        if (pos < shift) {
            src = 0;                                 // blocked below; value unused
        } else if (pos - shift >= sp) {
            src = hash_compress(a, b, pos - shift - sp);
        } else {
            src = a.cache[(int64_t)b * a.max_seq + (pos - shift)];
        }
        blocked = blocked || pos < shift || src == -1;
        const uint64_t term = (uint64_t)(blocked ? a.pad_id : src) * (uint64_t)m[shift];
        rolling = shift == 0 ? term : rolling ^ term;
    }
    const int64_t slot = (int64_t)li * C + col;
    return (int64_t)(rem_euclid_barrett(rolling, (uint64_t)a.primes[slot], a.bm[slot], a.wrap[slot]) +
                     (uint64_t)a.offsets[slot]);
}

// mbarrier phases with bounded waits (2 s on %globaltimer).
constexpr unsigned long long kWaitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// The same test, letting the thread sleep until the phase completes or about
// hint_ns pass (so a warp that waits long issues few instructions).
__device__ __forceinline__ bool mbar_try_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
// Bounded wait: false if the CTA is aborting or the wait ran out (then it
// raises the abort flag and the device error word).  sleep_ns > 0: each test
// may sleep that long (roles that wait for long stretches: the copy warp, the
// reducing warp).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          int *err, uint64_t limit_ns = kWaitNs, uint32_t sleep_ns = 0) {
    const uint64_t t0 = now_ns();
    while (!(sleep_ns ? mbar_try_sleep(bar, parity, sleep_ns) : mbar_try(bar, parity))) {
        if (*abort_flag) return false;
        if (now_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            set_err(err, ENGRAM_E_TIMEOUT);
            return false;
        }
    }
    return true;
}

// Programmatic dependent launch: wait for the grids this one depends on, and
// let the next grid in the stream start its independent prologue.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

struct RowsArgs {
    const uint8_t *table;   // fp8 codes [R, hd] or q2k blocks [R, 84]
    const void *scales;     // fp8: f32 or e8m0 bytes (fmt)
    int64_t R;
    int32_t hd, blk;
    const int64_t *ids;     // ids[t * id_stride + c]
    int64_t n_tok, id_stride;
    int32_t C;
    uint16_t *out;          // [n_tok * C, hd] bf16
    int *err;
    int32_t fmt;            // ENGRAM_FMT_FP8 or ENGRAM_FMT_FP8_E8M0 (fp8 rows)
};
cudaError_t launch_rows_fp8(const RowsArgs &a, cudaStream_t s);
cudaError_t launch_rows_q2k(const RowsArgs &a, cudaStream_t s);

// Hash and row gather (fp8 or Q2_K, the same format in every layer) of every
// layer in one launch: one lane hashes a row (its id written to hash.out, the
// cache written as the hash kernel does) and hands the id to the threads that
// gather the row.  layer[l]: table, scales, R, fmt and out (x of layer l);
// hd, blk and C from layer[0].
struct HashRowsArgs {
    RowsArgs layer[kMaxLayers];
    int32_t L;
    int64_t M;              // tokens (B * T)
};
bool hash_rows_supported(const HashRowsArgs &a);
cudaError_t launch_hash_rows(const HashRowsArgs &a, const HashArgs &h, cudaStream_t s);

// Small-T GEMV, optionally with the row gather fused into the x staging.
struct GemvLayer {
    const uint16_t *wkv;    // [N, K]
    const uint16_t *wkv_tiled;  // the same in 16 x 2048 tiles (engram_tile_wkv), or null
    const uint8_t *wkv_q2k; // [N, K / 256] Q2_K blocks (the q2k launch reads these instead)
    uint16_t *kv;           // [T, N]
    const uint16_t *x;      // plain x [T, K] (gather == 0)
    const uint8_t *table;   // gather source (gather == 1)
    const void *scales;     // f32 or e8m0 bytes, by fmt
    int64_t rows;
    const int64_t *ids;     // ids[t * id_stride + c] of this layer
    int32_t fmt;
};
struct GemvArgs {
    GemvLayer layer[kMaxLayers];
    int32_t L, T, K, N;
    int32_t hd, blk, C;
    int64_t id_stride;
    int32_t gather;
    int32_t fuse_hash;      // compute the row ids in-kernel (hash below), write them to ids_out
    HashArgs hash;          // hash.out = row ids [T, L, C] in the workspace
    int32_t pdl;            // launched as a programmatic dependent
    int *sched;             // per layer: next 16-row group, copy warps done (zero between launches), or null
    int *err;
};
constexpr int kFusedHashMaxIds = 2048;  // T * C row ids a CTA may hash for its layer
constexpr int kGemvMaxK = 6144;         // widest x the 1..8-token GEMV holds in registers
cudaError_t launch_gemv(const GemvArgs &a, cudaStream_t s);
cudaError_t launch_gemv_q2k(const GemvArgs &a, cudaStream_t s);   // one token, Q2_K wkv
size_t gemv_smem_bytes(int T, int K);
// wkv [N, K] -> 16-row x 2048-column tiles, g-major (the engram_tile_wkv layout).
constexpr int kTileRows = 16, kTileCols = 2048;
cudaError_t launch_tile_wkv(const uint16_t *wkv, int N, int K, uint16_t *tiled, cudaStream_t s);

// GEMM: kv [M, N] = bf16(x [M, K] . wkv [N, K]^T).
cudaError_t launch_gemm(const uint16_t *x, const uint16_t *wkv, uint16_t *kv, int M, int N, int K,
                        int *err, cudaStream_t s);
bool gemm_tc_supported(int M, int N, int K);
// Scratch that lets the CTA-pair GEMM cut the tiles of its partial last wave
// along K (engram_forward supplies it): f32 partial tiles, added up by a
// fix-up launch right after the GEMM.
constexpr int kTailItems = 96;                          // >= the CTA pairs of the GPU
constexpr size_t kTailPartBytes = (size_t)kTailItems * 256 * 256 * 4;
struct GemmTail {
    float *part;                                        // [kTailItems][256][256]
};
// pdl: launched as a programmatic dependent of the kernel before it (which
// writes x); the GEMM waits for it after its set-up (TMEM, barriers).  Pair
// kernel only (256 tokens and up), as is `tail`.
cudaError_t launch_gemm_tc(int L, const uint16_t *const *x, const uint16_t *const *wkv, uint16_t *const *kv,
                           int M, int N, int K, int *err, cudaStream_t s, bool pdl = false,
                           const GemmTail *tail = nullptr);
// The same on CTA pairs (tcgen05 cta_group::2, 256 x 256 tiles).
cudaError_t launch_gemm_tc2(int L, const uint16_t *const *x, const uint16_t *const *wkv, uint16_t *const *kv,
                           int M, int N, int K, int *err, cudaStream_t s, bool pdl = false,
                           const GemmTail *tail = nullptr);
cudaError_t launch_gemm_simt(const uint16_t *x, const uint16_t *wkv, uint16_t *kv, int M, int N,
                             int K, cudaStream_t s);

// Gate over several layers on one highway.
struct GateArgs {
    float *h;                           // [M, hc, D]
    int64_t *advance_pos;               // when set, block 0 adds advance_by once the projection is done
    int64_t advance_by;
    const uint16_t *kv[kMaxLayers];     // [M, (hc+1) D]
    const float *qk[kMaxLayers];        // [hc, D]
    int32_t L, M, hc, D;
    float eps, inv_sqrt_dim;
    int32_t pdl;            // launched as a programmatic dependent of the projection
};
cudaError_t launch_gate(const GateArgs &a, cudaStream_t s);

// Self-test of the bounded wait (selftest.cu): one wait that must run out.
cudaError_t launch_wait_timeout(int *err, uint64_t limit_ns, cudaStream_t s);

}  // namespace engram
