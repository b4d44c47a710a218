/*
 * engram.h -- C ABI of libengram, the GB300 (sm_103a) engram forward.
 *
 * The DeepSeek-V4.1 engram, per token and per engram layer (module docs of
 * "spark_model/layers/engram_v41.rs" and "Module engram_v41"):
 *   1. hash the n-gram window of compressed token ids into
 *      C = (max_ngram - 1) * n_heads row ids;
 *   2. gather and dequantise those C rows of the layer's table (fp8 e4m3 with
 *      power-of-two scales, or 84-byte Q2_K blocks) into x [C * head_dim];
 *   3. project kv = bf16(x . wkv^T), wkv [dim * (hc + 1), C * head_dim]:
 *      one key of dim per hyper-connection stream, then one shared value;
 *   4. gate: per stream c, s = <rmsnorm(h_c) (q k)_c, rmsnorm(key_c)> / sqrt(dim),
 *      g = sign(s) sqrt(max(|s|, 1e-6)), h_c += sigmoid(g) * value, in place
 *      on the FP32 highway h [tokens, hc, dim].
 *
 * Conventions for every entry point:
 *   - Pointers named d_* are DEVICE pointers, h_* are HOST pointers.  The
 *     caller owns every buffer it passes; the library keeps no pointer to it
 *     after the call returns, except the opaque handles it creates itself.
 *   - `stream` is a cudaStream_t passed as uintptr_t (0 = legacy default).
 *     Every compute call only enqueues work on that stream: no host
 *     synchronisation, no allocation, no host<->device copy (except
 *     engram_forward_host, which enqueues its own copies).
 *   - Return value: ENGRAM_OK (0) or a negative ENGRAM_E_* code.  Arguments
 *     are validated on the host before anything is enqueued; a call that
 *     returns an error has enqueued nothing.
 *   - Tables (fp8 codes and scales, Q2_K blocks) may live in device memory
 *     or in page-locked host memory that the device reads in place (mapped
 *     at the same address, e.g. cudaHostAlloc): rows are then read by id over
 *     the CPU-GPU link, so a table need not fit in HBM (the page-locked,
 *     device-visible arena of page "spark_model/layers/deepseek_v41_layer.rs").  Any
 *     other table pointer is refused with ENGRAM_E_INVALID.
 *   - T = 0 is a valid no-op for every call that takes a token count; its
 *     buffers may then be null.
 *   - Conditions only the device can see (a token id outside token_map, a
 *     row id outside a table) set a sticky per-device error word; the kernel
 *     substitutes a safe value (the token is treated as unmapped, the row as
 *     zeros) and never traps.  engram_check() synchronises the stream and
 *     returns and clears that word.
 */
#ifndef ENGRAM_H
#define ENGRAM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ENGRAM_OK 0
#define ENGRAM_E_INVALID -1     /* geometry or argument out of range */
#define ENGRAM_E_NULL -2        /* a required pointer is null */
#define ENGRAM_E_ALIGN -3       /* a pointer misses its required alignment */
#define ENGRAM_E_CAPACITY -4    /* start_pos + T exceeds the hasher's max_seq */
#define ENGRAM_E_WORKSPACE -5   /* workspace smaller than engram_workspace_bytes() */
#define ENGRAM_E_HC -6          /* hc outside 1..4 */
#define ENGRAM_E_TOKEN -7       /* device: an input token id outside token_map */
#define ENGRAM_E_ROW -8         /* device: a row id outside its table */
#define ENGRAM_E_CUDA -9        /* a CUDA runtime call failed */
#define ENGRAM_E_TIMEOUT -10    /* device: a bounded wait gave up */
#define ENGRAM_E_UNSUPPORTED -11 /* shape outside what the kernels handle */
#define ENGRAM_E_NOALLOC_LIMIT -12 /* request larger than engram_forward_noalloc's fixed scratch */

#define ENGRAM_FMT_FP8 0        /* e4m3 codes [rows, head_dim] + f32 scales [rows, head_dim / scale_block] */
#define ENGRAM_FMT_Q2K 1        /* 84-byte Q2_K super-blocks [rows, 84]; head_dim must be 256 */
#define ENGRAM_FMT_FP8_E8M0 2   /* e4m3 codes [rows, head_dim] + one-byte e8m0 scales [rows, head_dim / scale_block] */

/* Geometry.  C = (max_ngram - 1) * n_heads, K = C * head_dim, N = dim * (hc + 1).
 * Limits: 1 <= n_layers <= 4; 2 <= max_ngram <= 16; n_heads >= 1;
 * head_dim % 16 == 0, 16 <= head_dim <= 1024; scale_block % 16 == 0 and
 * divides head_dim; dim % 8 == 0, dim <= 16384; 1 <= hc <= 4
 * (EngramV41::new refuses other hc); vocab >= 1. */
typedef struct {
    int32_t n_layers, max_ngram, n_heads, head_dim, dim, hc, scale_block;
    int64_t vocab;
} engram_geom;

typedef struct engram_tables engram_tables;   /* device copies of the hash tables */
typedef struct engram_hasher engram_hasher;   /* per-batch look-back cache */

/* Hash tables: page "spark_model/layers/engram_v41.rs", module doc, item 1 (the
 * tables the hash reads; the ABI counterpart of `EngramHashTables::from_flat`).
 * Host arrays, copied to the current device:
 *   h_token_map   [vocab]                    compressed id per token, -1 = unmapped
 *   pad_token_id  pad_id = h_token_map[pad_token_id]
 *   h_multipliers [n_layers * max_ngram]     multipliers[layer][lookback]
 *   h_primes      [n_layers * C]             primes[layer][(ngram - 2) * n_heads + head]
 *   h_offsets     [n_layers * C]             offsets, same layout
 * Errors: ENGRAM_E_INVALID for bad geometry, pad_token_id outside token_map,
 * a multiplier/prime/offset above INT64_MAX or a prime of 0; ENGRAM_E_HC;
 * ENGRAM_E_CUDA if device allocation fails (set-up, not the hot path). */
int engram_tables_create(const engram_geom *geom, const int64_t *h_token_map,
                         int64_t pad_token_id, const uint64_t *h_multipliers,
                         const uint64_t *h_primes, const uint64_t *h_offsets,
                         engram_tables **out);
void engram_tables_destroy(engram_tables *t);

/* Look-back cache [batch, max_seq] of compressed ids, zero-filled like
 * `EngramHasher::new` / `NgramHashState::new`, so decode steps see the
 * prefill's ids.  The hasher borrows `t`, which must outlive it.  It also
 * holds the work counters of the 1..8-token projection (zero between
 * calls; one forward at a time on a hasher). */
int engram_hasher_create(const engram_tables *t, int32_t batch, int64_t max_seq,
                         engram_hasher **out);
/* `EngramHasher::reset`: the cache returns to zeros (enqueued on `stream`);
 * the projection's counters too (after ENGRAM_E_TIMEOUT they may not be). */
int engram_hasher_reset(engram_hasher *hs, uintptr_t stream);
void engram_hasher_destroy(engram_hasher *hs);

/* Stage 1, the hash: page "metrale_model_arch/deepseek_v41_ref/engram.rs", module
 * doc, item 1 (`EngramHasher::hash` / `NgramHashState::forward`):
 *   d_ids     [batch, T] int32 token ids at positions start_pos .. start_pos+T-1
 *   d_row_ids [batch, T, n_layers, C] int64 out
 * Writes the new positions into the cache.  The i64 arithmetic (wrapping
 * multiply, XOR roll, Euclidean remainder, + offset) is bit-exact.
 * Errors: ENGRAM_E_CAPACITY if start_pos + T > max_seq; device: ENGRAM_E_TOKEN. */
int engram_hash(engram_hasher *hs, const int32_t *d_ids, int32_t T, int64_t start_pos,
                int64_t *d_row_ids, uintptr_t stream);

/* Stage 2, fp8 rows (page "metrale_model_arch/deepseek_v41_ref/engram.rs", module
 * doc, item 2):
 *   row(id)[d] = bf16_rne(e4m3(d_table[id, d]) * d_scales[id, d / scale_block])
 * for id = d_row_ids[t * id_stride + c], written to d_rows[(t * C + c), :].
 *   d_table [R, head_dim] u8 (16-byte aligned), d_scales [R, head_dim/scale_block] f32,
 *   d_rows [n_tok * C, head_dim] bf16 (16-byte aligned).  Bit-exact. */
int engram_rows_fp8(const uint8_t *d_table, const float *d_scales, int64_t R, int32_t head_dim,
                    int32_t scale_block, const int64_t *d_row_ids, int64_t n_tok,
                    int64_t id_stride, int32_t C, uint16_t *d_rows, uintptr_t stream);

/* Stage 2, fp8 rows with one-byte scales: as engram_rows_fp8, with d_scales
 * [R, head_dim / scale_block] e8m0 bytes, scale = 2^(byte - 127) (the byte
 * `f32_to_e8m0_rne` on the CPU reference page stores; 255 is NaN).  Rows are
 * bit-identical to engram_rows_fp8 with the equal f32 scales. */
int engram_rows_fp8_e8m0(const uint8_t *d_table, const uint8_t *d_scales, int64_t R, int32_t head_dim,
                         int32_t scale_block, const int64_t *d_row_ids, int64_t n_tok, int64_t id_stride,
                         int32_t C, uint16_t *d_rows, uintptr_t stream);

/* Stage 2, Q2_K rows (page "spark_model/layers/engram_v41.rs", module doc, item 2;
 * head_dim 256): d_blocks [R, 84] u8 (4-byte aligned), ggml Q2_K layout,
 * decoded y = d * (sc & 15) * q - dmin * (sc >> 4), then bf16 RNE.  Bit-exact. */
int engram_rows_q2k(const uint8_t *d_blocks, int64_t R, const int64_t *d_row_ids, int64_t n_tok,
                    int64_t id_stride, int32_t C, uint16_t *d_rows, uintptr_t stream);

/* Stage 3 (page "metrale_model_arch/deepseek_v41_ref/engram.rs", module doc,
 * item 3): d_kv[t, o] =
 * bf16_rne(sum_i d_x[t, i] * d_wkv[o, i]) with f32 accumulation.
 *   d_x [T, K] bf16, d_wkv [N, K] bf16, d_kv [T, N] bf16; all 16-byte aligned.
 * K % 64 == 0, N % 16 == 0.  T <= 8 with K <= 6144 runs the bandwidth-bound
 * GEMV; otherwise the tcgen05 tensor-core GEMM, on CTA pairs (256 x 256 tiles)
 * from T = 256 and on single CTAs below, the two bit-identical. */
int engram_project(const uint16_t *d_x, const uint16_t *d_wkv, int32_t T, int32_t K, int32_t N,
                   uint16_t *d_kv, uintptr_t stream);

/* Stage 4 (page "metrale_model_arch/deepseek_v41_ref/engram.rs", module doc,
 * item 4, on the FP32 highway of page "spark_model/layers/engram_v41.rs",
 * module doc, item 4):
 *   d_h [T, hc, dim] f32 in/out (16-byte aligned); d_kv [T, (hc+1) dim] bf16;
 *   d_qk [hc, dim] f32 = q_weight * k_weight (exact for bf16 weights,
 *   `EngramV41::upload_qk`). */
int engram_gate(float *d_h, const uint16_t *d_kv, const float *d_qk, int32_t T, int32_t hc,
                int32_t dim, float eps, uintptr_t stream);

/* Stage 3 at one token from Q2_K-quantised wkv (page
 * "spark_model/layers/engram_v41.rs", the doc of the layer weights: the weight
 * as the GGUF ships it, read by the
 * single-token projection in place of the bf16 expansion, 6x fewer bytes):
 *   d_wkv_q2k [N, K / 256] 84-byte ggml Q2_K blocks (a row's blocks contiguous,
 *   16-byte aligned); d_x [1, K] bf16; d_kv [1, N] bf16.  K % 256 == 0 and
 *   K <= 6144 (ENGRAM_E_UNSUPPORTED above).
 * kv is bit-identical to engram_project(d_x, W) where W is the bf16
 * dequantisation of the blocks (engram_rows_q2k). */
int engram_project_q2k(const uint16_t *d_x, const uint8_t *d_wkv_q2k, int32_t K, int32_t N,
                       uint16_t *d_kv, uintptr_t stream);

/* wkv tiled for the 1..8-token projection (a layout of the same weights,
 * made once when the weights are loaded; not a step of the method).  Tile
 * (g, c) holds rows 16 g .. 16 g + 15 and columns 2048 c .. 2048 c + 2047 of
 * wkv [N, K] bf16, row after row, 64 KB contiguous; tiles are ordered g-major:
 *   tiled[((g * ceil(K / 2048) + c) * 16 + r) * 2048 + j] = wkv[16 g + r, 2048 c + j],
 * zero where 16 g + r >= N or 2048 c + j >= K.  The projection then streams
 * each 16-row group's pieces from one contiguous range instead of 16 rows
 * 2 K bytes apart.  engram_tiled_wkv_bytes gives the size; engram_tile_wkv writes
 * it (d_wkv and d_tiled device memory, 16-byte aligned, not overlapping;
 * stream-ordered, no host sync). */
size_t engram_tiled_wkv_bytes(int32_t N, int32_t K);
int engram_tile_wkv(const uint16_t *d_wkv, int32_t N, int32_t K, uint16_t *d_tiled, uintptr_t stream);

/* One engram layer for engram_forward. */
typedef struct {
    const void *table;      /* FP8, FP8_E8M0: e4m3 [rows, head_dim]; Q2K: blocks [rows, 84] */
    const void *scales;     /* FP8: f32 [rows, head_dim / scale_block]; FP8_E8M0: e8m0 bytes,
                               same shape; Q2K: unused */
    int64_t rows;           /* table rows (sum of the layer's primes) */
    int32_t fmt;            /* ENGRAM_FMT_FP8, ENGRAM_FMT_Q2K or ENGRAM_FMT_FP8_E8M0 */
    const uint16_t *wkv;    /* [dim * (hc + 1), C * head_dim] bf16; may be NULL when wkv_q2k
                               is set and every call has batch * T <= 8 */
    const float *qk;        /* [hc, dim] f32 */
    const uint8_t *wkv_q2k; /* optional [dim * (hc + 1), C * head_dim / 256] Q2_K blocks,
                               16-byte aligned: when every layer has it and C * head_dim
                               <= 6144, calls of 1..8 tokens (batch * T) project from it,
                               bit-identical to the bf16 path on the dequantised blocks */
    const uint16_t *wkv_tiled; /* optional engram_tile_wkv(wkv), 16-byte aligned: calls of
                               1..8 tokens that project from bf16 read the layer's weights
                               from it instead of wkv, with bit-identical results; wkv is
                               still required (the larger calls read it) */
} engram_layer;

/* The whole forward for n_layers engram layers (in `layers` order) on one
 * highway, every layer hashed together (as `V41Runtime.step_hashes` reuses
 * them).  Up to 8 tokens (batch * T) with C * head_dim <= 6144: one launch
 * hashes, gathers and projects every layer, then one launch applies every
 * layer's gate.  Larger calls: one launch hashes and gathers the rows of
 * every layer (when every layer's table has the same format and, for fp8,
 * head_dim / 16 and scale_block are powers of two; otherwise the hash launch
 * and one row-gather launch per layer), one tensor-core GEMM launch for every
 * layer, then the gates.
 *   d_ids [batch, T] int32 at positions start_pos..; d_h [batch * T, hc, dim]
 *   f32 in/out; d_ws device workspace of at least
 *   engram_workspace_bytes(geom, batch * T) bytes, 256-byte aligned.
 * After the call the workspace holds (offsets from engram_workspace_layout):
 *   row ids [batch*T, n_layers, C] int64, then per layer kv [batch*T, N] bf16. */
int engram_forward(engram_hasher *hs, const engram_layer *layers, const int32_t *d_ids,
                   int32_t T, int64_t start_pos, float *d_h, float eps, void *d_ws,
                   size_t ws_bytes, uintptr_t stream);

/* engram_forward with the start position in device memory: *d_start_pos
 * (int64, 8-byte aligned) is read on the device and advanced by T when the
 * step's last kernel runs, so consecutive calls -- or replays of a captured
 * graph -- walk the sequence without the host.  A position past the cache is
 * reported on the device (ENGRAM_E_CAPACITY through engram_check) and the
 * step touches no cache entry. */
int engram_forward_dpos(engram_hasher *hs, const engram_layer *layers, const int32_t *d_ids, int32_t T,
                        int64_t *d_start_pos, float *d_h, float eps, void *d_ws, size_t ws_bytes,
                        uintptr_t stream);

/* The decode step as one CUDA graph (the single-token step capture of
 * page "spark_model/layers/deepseek_v41_layer.rs", the doc of its graph mode): captures
 * engram_forward_dpos with these arguments -- every pointer is baked into the
 * graph -- and replays it with engram_graph_launch.  Between replays the
 * caller updates the contents of d_ids (and of d_h if it wishes); the
 * position advances by itself.  Replays give bit-identical results to eager
 * engram_forward calls at the same positions. */
typedef struct engram_graph engram_graph;
int engram_graph_create(engram_hasher *hs, const engram_layer *layers, const int32_t *d_ids, int32_t T,
                        int64_t *d_start_pos, float *d_h, float eps, void *d_ws, size_t ws_bytes,
                        engram_graph **out);
/* The same for `steps` consecutive decode steps in one graph (1 <= steps <=
 * 4096, steps * T <= max_seq): d_ids [steps, batch, T] and d_h [steps,
 * batch * T, hc, dim], step k reading ids k and updating highway rows k at
 * position *d_start_pos + k T; the last step's gate advances the position by
 * steps * T.  Inside a replay the steps overlap as eager calls do (each step's
 * hash, row gather and wkv stream run beside the previous step's gate), so one
 * replay costs about `steps` eager steps plus one graph launch.  Replays give
 * bit-identical results to `steps` eager engram_forward calls at the same
 * positions.  engram_graph_create is this with steps = 1. */
int engram_graph_create_steps(engram_hasher *hs, const engram_layer *layers, const int32_t *d_ids, int32_t T,
                              int32_t steps, int64_t *d_start_pos, float *d_h, float eps, void *d_ws,
                              size_t ws_bytes, engram_graph **out);
int engram_graph_launch(engram_graph *g, uintptr_t stream);
void engram_graph_destroy(engram_graph *g);

/* engram_forward from host buffers h_ids [batch, T] and h_h [batch*T, hc, dim]
 * (in/out).  When both are page-locked and mapped for the device (e.g.
 * cudaHostAlloc), the kernels read the ids and update the highway in place
 * over the CPU-GPU link and d_ids / d_h are not used.  Otherwise the call
 * enqueues the copies into the device staging buffers d_ids / d_h, the
 * forward and the copy of d_h back into h_h; the highway upload then runs on
 * the hasher's own auxiliary stream (created with the hasher), ordered after
 * the caller's earlier work, so it overlaps the projection.  Either way the
 * caller synchronises `stream` before reading h_h. */
int engram_forward_host(engram_hasher *hs, const engram_layer *layers, const int32_t *h_ids,
                        int32_t *d_ids, int32_t T, int64_t start_pos, float *h_h, float *d_h,
                        float eps, void *d_ws, size_t ws_bytes, uintptr_t stream);

/* engram_forward for callers that cannot allocate device memory.  (The pages
 * have no counterpart: this entry point belongs to this library's ABI.)
 * Code that runs where cudaMalloc is unavailable or unwelcome -- inside a host
 * that owns every allocation itself, a real-time loop that must not enter the
 * allocator, or a plugin with no allocator handle -- still needs the forward's
 * scratch (row ids and per-layer kv, plus the gathered rows beyond 8 tokens).
 * This entry point takes it from a fixed 4 MiB array that the library places
 * in device memory (a file-scope __device__ array, held on every GPU that
 * loads the library until the process exits), so the call allocates nothing.
 *   Arguments and results are those of engram_forward without d_ws/ws_bytes.
 *   A request whose workspace (engram_workspace_bytes for batch * T tokens)
 *   exceeds 4 MiB is refused with ENGRAM_E_NOALLOC_LIMIT before anything is
 *   enqueued; at the V4.1-Flash shape that is about 39 tokens a call.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 *   Every call on a device shares the one array, which keeps the previous
 *   call's contents (nothing in it needs to start at zero: each call writes
 *   what it reads).  Calls whose work overlaps on the GPU -- on different
 *   streams, or from different threads -- race on it: serialise them. */
int engram_forward_noalloc(engram_hasher *hs, const engram_layer *layers, const int32_t *d_ids,
                           int32_t T, int64_t start_pos, float *d_h, float eps, uintptr_t stream);

/* Workspace bytes engram_forward needs for up to max_tokens = batch * T. */
size_t engram_workspace_bytes(const engram_geom *geom, int64_t max_tokens);

/* Byte offsets inside the workspace for `tokens` tokens: off[0] = row ids,
 * off[1 + l] = kv of layer l, off[1 + n_layers + l] = gathered rows x of
 * layer l (present only when the projection runs as a GEMM: tokens > 8, or
 * C * head_dim > 6144), off[1 + 2 n_layers] = total bytes.  From 256 tokens
 * the total also covers, at the end, 24 MiB of f32 partial tiles for the
 * tensor-core GEMM's last wave, which it may cut along K (the tiles of that
 * wave are then summed from K ranges in a fixed order: deterministic, but not
 * bit-identical to the unsplit accumulation).
 * off must hold 2 + 2 * n_layers entries. */
int engram_workspace_layout(const engram_geom *geom, int64_t tokens, size_t *off);

/* Optional stage timing: when set, engram_forward records on its stream
 * events[0] before the hash, [1] after it (== [0] where the hash runs inside
 * the next launch), [2] after the row gather (== [1] where the gather is
 * fused into the projection), [3] after the projection and [4] after the
 * gate.  The events sit between the launches, so a profiled step loses the
 * overlap of programmatic launches.  events holds 5 cudaEvent_t as uintptr_t; the
 * library keeps the pointer (the array must stay alive) until it is set to
 * NULL.  Process-wide; not thread-safe. */
int engram_set_profile_events(const uintptr_t *events, int32_t n);

/* Synchronises `stream`, then returns and clears the current device's
 * sticky error word (ENGRAM_OK if none). */
int engram_check(uintptr_t stream);

/* Self-test of failure detection (not a step of the method): enqueues one
 * kernel whose thread waits, through the same bounded mbarrier wait that
 * every copy ring and GEMM here uses, on a barrier nothing arrives at, for
 * limit_us microseconds (1 .. 1e6); the wait gives up, the kernel raises
 * ENGRAM_E_TIMEOUT in the error word (read by engram_check) and returns, and
 * the device stays usable.  ENGRAM_E_INVALID for a limit out of range. */
int engram_selftest_wait_timeout(int32_t limit_us, uintptr_t stream);

const char *engram_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* ENGRAM_H */
