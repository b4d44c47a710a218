// api.cu -- the libengram C ABI: handles, host-side validation (before any
// copy or launch, as the GPU module page "spark_model/layers/engram_v41.rs"
// checks its shapes before it uploads or launches), and the launch sequence of
// the forward.
#include "common.cuh"

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

using namespace engram;

struct engram_tables {
    engram_geom g;
    int64_t pad_id;
    int device;
    int64_t *token_map, *mult, *primes, *offsets;
    uint64_t *bm, *wrap;      // Barrett constants of the primes (see rem_euclid_barrett)
};

struct engram_hasher {
    const engram_tables *t;
    int32_t batch;
    int64_t max_seq;
    int64_t *cache;
    int *sched;             // the projection's work counters, 2 a layer, zero between launches
    int device;
    // engram_forward_host: the highway upload runs on `aux` while the
    // projection streams wkv on the caller's stream; only the gate waits.
    cudaStream_t aux;
    cudaEvent_t ev_main, ev_h;
};

namespace engram {
// Geometry and batch of a hasher, for entry points defined in other files.
bool hasher_geometry(const engram_hasher *hs, engram_geom *g, int *batch) {
    if (!hs || !hs->t) return false;
    *g = hs->t->g;
    *batch = hs->batch;
    return true;
}
}  // namespace engram

// The sticky error word, one per device (this module's copy on each GPU).
static __device__ int g_err_word;

namespace {

std::mutex g_mu;
int *g_err_ptr[64] = {};
const uintptr_t *g_prof_events = nullptr;

int *err_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<int *>(p);
    }
    return g_err_ptr[dev];
}

inline cudaStream_t S(uintptr_t s) { return reinterpret_cast<cudaStream_t>(s); }
inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

inline int cols(const engram_geom &g) { return (g.max_ngram - 1) * g.n_heads; }

int check_geom(const engram_geom *g) {
    if (!g) return ENGRAM_E_NULL;
    if (g->hc < 1 || g->hc > 4) return ENGRAM_E_HC;
    if (g->n_layers < 1 || g->n_layers > kMaxLayers) return ENGRAM_E_INVALID;
    if (g->max_ngram < 2 || g->max_ngram > kMaxNgram) return ENGRAM_E_INVALID;
    if (g->n_heads < 1 || g->n_heads > 1024) return ENGRAM_E_INVALID;
    if (g->head_dim < 16 || g->head_dim > 1024 || g->head_dim % 16) return ENGRAM_E_INVALID;
    if (g->scale_block < 16 || g->scale_block % 16 || g->head_dim % g->scale_block) return ENGRAM_E_INVALID;
    if (g->dim < 8 || g->dim % 8 || g->dim > 16384) return ENGRAM_E_INVALID;
    if (g->vocab < 1) return ENGRAM_E_INVALID;
    const int64_t K = (int64_t)cols(*g) * g->head_dim;
    if (K % 64 || K > (1 << 20)) return ENGRAM_E_UNSUPPORTED;
    return ENGRAM_OK;
}

void record(int i, cudaStream_t s) {
    if (g_prof_events) cudaEventRecord(reinterpret_cast<cudaEvent_t>(g_prof_events[i]), s);
}

inline int cuda_rc(cudaError_t e) { return e == cudaSuccess ? ENGRAM_OK : ENGRAM_E_CUDA; }

template <class T>
int dev_copy(T **dst, const T *src, size_t n) {
    *dst = nullptr;
    if (cudaMalloc(reinterpret_cast<void **>(dst), n * sizeof(T) + 16) != cudaSuccess) return ENGRAM_E_CUDA;
    if (cudaMemcpy(*dst, src, n * sizeof(T), cudaMemcpyHostToDevice) != cudaSuccess) return ENGRAM_E_CUDA;
    return ENGRAM_OK;
}

// Tables may live in device memory or in page-locked host memory the device
// reads in place (mapped, same address); anything else would fault the GPU,
// so it is refused before any launch.
bool device_readable(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return true;
    if (at.type == cudaMemoryTypeHost) return at.devicePointer == p;
    return false;
}

// The projection of one layer's x [M, K] (or of its fused gather) into kv.
bool gemv_fits(int M, int K) {
    return M >= 1 && M <= kSmallT && gemv_smem_bytes(M, K) != SIZE_MAX;
}

}  // namespace

extern "C" {

const char *engram_strerror(int code) {
    switch (code) {
        case ENGRAM_OK: return "ok";
        case ENGRAM_E_INVALID: return "geometry or argument out of range";
        case ENGRAM_E_NULL: return "a required pointer is null";
        case ENGRAM_E_ALIGN: return "a pointer misses its required alignment";
        case ENGRAM_E_CAPACITY: return "start_pos + T exceeds the hasher's max_seq";
        case ENGRAM_E_WORKSPACE: return "workspace smaller than engram_workspace_bytes()";
        case ENGRAM_E_HC: return "engram gate supports hc 1..4";
        case ENGRAM_E_TOKEN: return "a token id outside the engram token_map";
        case ENGRAM_E_ROW: return "a row id outside its engram table";
        case ENGRAM_E_CUDA: return "a CUDA runtime call failed";
        case ENGRAM_E_TIMEOUT: return "a bounded device wait gave up";
        case ENGRAM_E_UNSUPPORTED: return "shape outside what the kernels handle";
        case ENGRAM_E_NOALLOC_LIMIT: return "request larger than the fixed scratch of engram_forward_noalloc";
        default: return "unknown engram error";
    }
}

int engram_tables_create(const engram_geom *geom, const int64_t *h_token_map, int64_t pad_token_id,
                         const uint64_t *h_multipliers, const uint64_t *h_primes,
                         const uint64_t *h_offsets, engram_tables **out) {
    if (!out) return ENGRAM_E_NULL;
    *out = nullptr;
    int rc = check_geom(geom);
    if (rc) return rc;
    if (!h_token_map || !h_multipliers || !h_primes || !h_offsets) return ENGRAM_E_NULL;
    const engram_geom g = *geom;
    if (pad_token_id < 0 || pad_token_id >= g.vocab) return ENGRAM_E_INVALID;
    const size_t nm = (size_t)g.n_layers * g.max_ngram, nc = (size_t)g.n_layers * cols(g);
    for (size_t i = 0; i < nm; ++i)
        if (h_multipliers[i] > (uint64_t)INT64_MAX) return ENGRAM_E_INVALID;
    for (size_t i = 0; i < nc; ++i)
        if (h_primes[i] == 0 || h_primes[i] > (uint64_t)INT64_MAX || h_offsets[i] > (uint64_t)INT64_MAX)
            return ENGRAM_E_INVALID;
    engram_tables *t = new engram_tables();
    t->g = g;
    t->pad_id = h_token_map[pad_token_id];
    cudaGetDevice(&t->device);
    rc = dev_copy(&t->token_map, h_token_map, (size_t)g.vocab);
    if (!rc) rc = dev_copy(&t->mult, reinterpret_cast<const int64_t *>(h_multipliers), nm);
    if (!rc) rc = dev_copy(&t->primes, reinterpret_cast<const int64_t *>(h_primes), nc);
    if (!rc) rc = dev_copy(&t->offsets, reinterpret_cast<const int64_t *>(h_offsets), nc);
    if (!rc) {
        std::vector<uint64_t> bm(nc), wrap(nc);
        for (size_t i = 0; i < nc; ++i) {
            const unsigned __int128 two64 = (unsigned __int128)1 << 64;
            bm[i] = h_primes[i] == 1 ? 0 : (uint64_t)(two64 / h_primes[i]);
            wrap[i] = (uint64_t)(two64 % h_primes[i]);
        }
        rc = dev_copy(&t->bm, bm.data(), nc);
        if (!rc) rc = dev_copy(&t->wrap, wrap.data(), nc);
    }
    if (rc) {
        engram_tables_destroy(t);
        return rc;
    }
    *out = t;
    return ENGRAM_OK;
}

void engram_tables_destroy(engram_tables *t) {
    if (!t) return;
    cudaFree(t->token_map);
    cudaFree(t->mult);
    cudaFree(t->primes);
    cudaFree(t->offsets);
    cudaFree(t->bm);
    cudaFree(t->wrap);
    delete t;
}

int engram_hasher_create(const engram_tables *t, int32_t batch, int64_t max_seq, engram_hasher **out) {
    if (!out || !t) return ENGRAM_E_NULL;
    *out = nullptr;
    if (batch < 1 || max_seq < 1 || max_seq > (int64_t(1) << 40) / batch) return ENGRAM_E_INVALID;
    engram_hasher *h = new engram_hasher();
    h->t = t;
    h->batch = batch;
    h->max_seq = max_seq;
    cudaGetDevice(&h->device);
    const size_t bytes = (size_t)batch * max_seq * sizeof(int64_t);
    const size_t sched_bytes = 2 * kMaxLayers * sizeof(int);
    if (cudaMalloc(&h->cache, bytes) != cudaSuccess || cudaMemset(h->cache, 0, bytes) != cudaSuccess ||
        cudaMalloc(&h->sched, sched_bytes) != cudaSuccess || cudaMemset(h->sched, 0, sched_bytes) != cudaSuccess ||
        cudaStreamCreateWithFlags(&h->aux, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_main, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_h, cudaEventDisableTiming) != cudaSuccess) {
        engram_hasher_destroy(h);
        return ENGRAM_E_CUDA;
    }
    if (!err_ptr()) {
        engram_hasher_destroy(h);
        return ENGRAM_E_CUDA;
    }
    *out = h;
    return ENGRAM_OK;
}

int engram_hasher_reset(engram_hasher *hs, uintptr_t stream) {
    if (!hs) return ENGRAM_E_NULL;
    if (cudaMemsetAsync(hs->sched, 0, 2 * kMaxLayers * sizeof(int), S(stream)) != cudaSuccess) return ENGRAM_E_CUDA;
    return cuda_rc(cudaMemsetAsync(hs->cache, 0, (size_t)hs->batch * hs->max_seq * sizeof(int64_t), S(stream)));
}

void engram_hasher_destroy(engram_hasher *hs) {
    if (!hs) return;
    cudaFree(hs->cache);
    cudaFree(hs->sched);
    if (hs->ev_h) cudaEventDestroy(hs->ev_h);
    if (hs->ev_main) cudaEventDestroy(hs->ev_main);
    if (hs->aux) cudaStreamDestroy(hs->aux);
    delete hs;
}

int engram_set_profile_events(const uintptr_t *events, int32_t n) {
    if (events && n < 5) return ENGRAM_E_INVALID;
    g_prof_events = events;
    return ENGRAM_OK;
}

int engram_check(uintptr_t stream) {
    if (cudaStreamSynchronize(S(stream)) != cudaSuccess) return ENGRAM_E_CUDA;
    int *p = err_ptr();
    if (!p) return ENGRAM_E_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ENGRAM_E_CUDA;
    if (v != 0 && cudaMemset(p, 0, sizeof(int)) != cudaSuccess) return ENGRAM_E_CUDA;
    return v;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Compute entry points
// ---------------------------------------------------------------------------
namespace {

HashArgs hash_args(engram_hasher *hs, const int32_t *d_ids, int32_t T, int64_t start_pos,
                   int64_t *d_row_ids, const int64_t *d_pos = nullptr, bool pos_stable = false) {
    const engram_tables *t = hs->t;
    HashArgs a;
    a.ids = d_ids;
    a.B = hs->batch;
    a.T = T;
    a.start_pos = start_pos;
    a.start_pos_dev = d_pos;
    a.pos_stable = pos_stable ? 1 : 0;
    a.token_map = t->token_map;
    a.vocab = t->g.vocab;
    a.pad_id = t->pad_id;
    a.mult = t->mult;
    a.primes = t->primes;
    a.offsets = t->offsets;
    a.bm = t->bm;
    a.wrap = t->wrap;
    a.L = t->g.n_layers;
    a.ng = t->g.max_ngram;
    a.H = t->g.n_heads;
    a.cache = hs->cache;
    a.max_seq = hs->max_seq;
    a.out = d_row_ids;
    a.err = err_ptr();
    return a;
}

int check_hash(engram_hasher *hs, const int32_t *d_ids, int32_t T, int64_t start_pos, const void *out) {
    if (!hs) return ENGRAM_E_NULL;
    if (T < 0 || start_pos < 0) return ENGRAM_E_INVALID;
    if (start_pos + T > hs->max_seq) return ENGRAM_E_CAPACITY;
    if (T == 0) return ENGRAM_OK;                 // nothing to read or write
    if (!d_ids || !out) return ENGRAM_E_NULL;
    if (!aligned(d_ids, 4) || !aligned(out, 8)) return ENGRAM_E_ALIGN;
    return ENGRAM_OK;
}

int check_rows(const uint8_t *table, const int64_t *ids, int64_t R, int64_t n_tok, int64_t id_stride,
               int32_t C, const uint16_t *rows) {
    if (!table || !ids || !rows) return ENGRAM_E_NULL;
    if (R < 1 || n_tok < 0 || C < 1 || id_stride < C) return ENGRAM_E_INVALID;
    if (!aligned(ids, 8) || !aligned(rows, 16)) return ENGRAM_E_ALIGN;
    return ENGRAM_OK;
}

}  // namespace

extern "C" {

int engram_hash(engram_hasher *hs, const int32_t *d_ids, int32_t T, int64_t start_pos,
                int64_t *d_row_ids, uintptr_t stream) {
    int rc = check_hash(hs, d_ids, T, start_pos, d_row_ids);
    if (rc || T == 0) return rc;
    if (!err_ptr()) return ENGRAM_E_CUDA;
    return cuda_rc(launch_hash(hash_args(hs, d_ids, T, start_pos, d_row_ids), S(stream)));
}

int engram_rows_fp8(const uint8_t *d_table, const float *d_scales, int64_t R, int32_t head_dim,
                    int32_t scale_block, const int64_t *d_row_ids, int64_t n_tok, int64_t id_stride,
                    int32_t C, uint16_t *d_rows, uintptr_t stream) {
    int rc = check_rows(d_table, d_row_ids, R, n_tok, id_stride, C, d_rows);
    if (rc) return rc;
    if (!d_scales) return ENGRAM_E_NULL;
    if (head_dim < 16 || head_dim > 1024 || head_dim % 16 || scale_block < 16 || scale_block % 16 ||
        head_dim % scale_block)
        return ENGRAM_E_INVALID;
    if (!aligned(d_table, 16) || !aligned(d_scales, 4)) return ENGRAM_E_ALIGN;
    if (!device_readable(d_table) || !device_readable(d_scales)) return ENGRAM_E_INVALID;
    RowsArgs a{d_table, d_scales, R, head_dim, scale_block, d_row_ids, n_tok, id_stride, C, d_rows, err_ptr(),
               ENGRAM_FMT_FP8};
    if (!a.err) return ENGRAM_E_CUDA;
    return cuda_rc(launch_rows_fp8(a, S(stream)));
}

int engram_rows_fp8_e8m0(const uint8_t *d_table, const uint8_t *d_scales, int64_t R, int32_t head_dim,
                         int32_t scale_block, const int64_t *d_row_ids, int64_t n_tok, int64_t id_stride,
                         int32_t C, uint16_t *d_rows, uintptr_t stream) {
    int rc = check_rows(d_table, d_row_ids, R, n_tok, id_stride, C, d_rows);
    if (rc) return rc;
    if (!d_scales) return ENGRAM_E_NULL;
    if (head_dim < 16 || head_dim > 1024 || head_dim % 16 || scale_block < 16 || scale_block % 16 ||
        head_dim % scale_block)
        return ENGRAM_E_INVALID;
    if (!aligned(d_table, 16)) return ENGRAM_E_ALIGN;
    if (!device_readable(d_table) || !device_readable(d_scales)) return ENGRAM_E_INVALID;
    RowsArgs a{d_table, d_scales, R, head_dim, scale_block, d_row_ids, n_tok, id_stride, C, d_rows, err_ptr(),
               ENGRAM_FMT_FP8_E8M0};
    if (!a.err) return ENGRAM_E_CUDA;
    return cuda_rc(launch_rows_fp8(a, S(stream)));
}

int engram_rows_q2k(const uint8_t *d_blocks, int64_t R, const int64_t *d_row_ids, int64_t n_tok,
                    int64_t id_stride, int32_t C, uint16_t *d_rows, uintptr_t stream) {
    int rc = check_rows(d_blocks, d_row_ids, R, n_tok, id_stride, C, d_rows);
    if (rc) return rc;
    if (!aligned(d_blocks, 4)) return ENGRAM_E_ALIGN;
    if (!device_readable(d_blocks)) return ENGRAM_E_INVALID;
    RowsArgs a{d_blocks, nullptr, R, 256, 256, d_row_ids, n_tok, id_stride, C, d_rows, err_ptr(), ENGRAM_FMT_Q2K};
    if (!a.err) return ENGRAM_E_CUDA;
    return cuda_rc(launch_rows_q2k(a, S(stream)));
}

int engram_project(const uint16_t *d_x, const uint16_t *d_wkv, int32_t T, int32_t K, int32_t N,
                   uint16_t *d_kv, uintptr_t stream) {
    if (!d_x || !d_wkv || !d_kv) return ENGRAM_E_NULL;
    if (T < 0 || K < 64 || K % 64 || N < 16 || N % 16) return ENGRAM_E_INVALID;
    if (!aligned(d_x, 16) || !aligned(d_wkv, 16) || !aligned(d_kv, 16)) return ENGRAM_E_ALIGN;
    if (T == 0) return ENGRAM_OK;
    int *err = err_ptr();
    if (!err) return ENGRAM_E_CUDA;
    if (gemv_fits(T, K)) {
        GemvArgs a{};
        a.layer[0].wkv = d_wkv;
        a.layer[0].kv = d_kv;
        a.layer[0].x = d_x;
        a.L = 1;
        a.T = T;
        a.K = K;
        a.N = N;
        a.gather = 0;
        a.err = err;
        return cuda_rc(launch_gemv(a, S(stream)));
    }
    return cuda_rc(launch_gemm(d_x, d_wkv, d_kv, T, N, K, err, S(stream)));
}

int engram_project_q2k(const uint16_t *d_x, const uint8_t *d_wkv_q2k, int32_t K, int32_t N, uint16_t *d_kv,
                       uintptr_t stream) {
    if (!d_x || !d_wkv_q2k || !d_kv) return ENGRAM_E_NULL;
    if (K < 256 || K % 256 || N < 1 || K > (1 << 20)) return ENGRAM_E_INVALID;
    if (!aligned(d_x, 16) || !aligned(d_wkv_q2k, 16) || !aligned(d_kv, 2)) return ENGRAM_E_ALIGN;
    if (K > kGemvMaxK) return ENGRAM_E_UNSUPPORTED;
    int *err = err_ptr();
    if (!err) return ENGRAM_E_CUDA;
    GemvArgs a{};
    a.layer[0].wkv_q2k = d_wkv_q2k;
    a.layer[0].kv = d_kv;
    a.layer[0].x = d_x;
    a.L = 1;
    a.T = 1;
    a.K = K;
    a.N = N;
    a.gather = 0;
    a.err = err;
    return cuda_rc(launch_gemv_q2k(a, S(stream)));
}

int engram_selftest_wait_timeout(int32_t limit_us, uintptr_t stream) {
    if (limit_us < 1 || limit_us > 1000000) return ENGRAM_E_INVALID;
    int *err = err_ptr();
    if (!err) return ENGRAM_E_CUDA;
    return cuda_rc(launch_wait_timeout(err, (uint64_t)limit_us * 1000ull, S(stream)));
}

size_t engram_tiled_wkv_bytes(int32_t N, int32_t K) {
    if (N < 1 || K < 8 || K % 8) return 0;
    const size_t groups = ((size_t)N + kTileRows - 1) / kTileRows, chunks = ((size_t)K + kTileCols - 1) / kTileCols;
    return groups * chunks * kTileRows * kTileCols * sizeof(uint16_t);
}

int engram_tile_wkv(const uint16_t *d_wkv, int32_t N, int32_t K, uint16_t *d_tiled, uintptr_t stream) {
    if (!d_wkv || !d_tiled) return ENGRAM_E_NULL;
    if (N < 1 || K < 8 || K % 8) return ENGRAM_E_INVALID;
    if (!aligned(d_wkv, 16) || !aligned(d_tiled, 16)) return ENGRAM_E_ALIGN;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(d_wkv), a1 = a0 + (size_t)N * K * 2;
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(d_tiled), b1 = b0 + engram_tiled_wkv_bytes(N, K);
    if (a0 < b1 && b0 < a1) return ENGRAM_E_INVALID;        // overlapping buffers
    return cuda_rc(launch_tile_wkv(d_wkv, N, K, d_tiled, S(stream)));
}

int engram_gate(float *d_h, const uint16_t *d_kv, const float *d_qk, int32_t T, int32_t hc, int32_t dim,
                float eps, uintptr_t stream) {
    if (!d_h || !d_kv || !d_qk) return ENGRAM_E_NULL;
    if (hc < 1 || hc > 4) return ENGRAM_E_HC;
    if (T < 0 || dim < 8 || dim % 8 || dim > 16384 || !(eps >= 0.0f)) return ENGRAM_E_INVALID;
    if (!aligned(d_h, 16) || !aligned(d_kv, 16) || !aligned(d_qk, 16)) return ENGRAM_E_ALIGN;
    GateArgs a{};
    a.h = d_h;
    a.kv[0] = d_kv;
    a.qk[0] = d_qk;
    a.L = 1;
    a.M = T;
    a.hc = hc;
    a.D = dim;
    a.eps = eps;
    a.inv_sqrt_dim = powf((float)dim, -0.5f);
    return cuda_rc(launch_gate(a, S(stream)));
}

int engram_workspace_layout(const engram_geom *geom, int64_t tokens, size_t *off) {
    int rc = check_geom(geom);
    if (rc) return rc;
    if (!off) return ENGRAM_E_NULL;
    if (tokens < 0) return ENGRAM_E_INVALID;
    const engram_geom &g = *geom;
    const size_t C = (size_t)cols(g), K = C * g.head_dim, N = (size_t)g.dim * (g.hc + 1);
    size_t p = 0;
    off[0] = p;
    p += up256((size_t)tokens * g.n_layers * C * sizeof(int64_t));
    for (int l = 0; l < g.n_layers; ++l) {
        off[1 + l] = p;
        p += up256((size_t)tokens * N * 2);
    }
    const bool need_x = !gemv_fits((int)(tokens > kSmallT ? kSmallT + 1 : tokens), (int)K);
    for (int l = 0; l < g.n_layers; ++l) {
        off[1 + g.n_layers + l] = p;
        if (need_x) p += up256((size_t)tokens * K * 2);
    }
    // from 256 tokens (the CTA-pair GEMM): partial tiles of its last wave, at the end
    if (tokens >= 256) p += up256(kTailPartBytes);
    off[1 + 2 * g.n_layers] = p;   // total (caller's array is sized 2 + 2 L by engram_workspace_bytes)
    return ENGRAM_OK;
}

size_t engram_workspace_bytes(const engram_geom *geom, int64_t max_tokens) {
    size_t off[2 + 2 * kMaxLayers];
    if (engram_workspace_layout(geom, max_tokens, off) != ENGRAM_OK) return 0;
    return off[1 + 2 * geom->n_layers];
}

}  // extern "C"

namespace {

// How a step reads a device-resident position: at *d_pos + offset; the step's
// gate then adds advance (0: leaves it); stable: nothing writes it before
// this step's own gate.
struct DevPos {
    int64_t offset, advance;
    bool stable;
};

// The forward; d_pos (device memory) replaces start_pos when set, and is then
// advanced by T at the end of the step (or as `dp` says).
int forward_impl(engram_hasher *hs, const engram_layer *layers, const int32_t *d_ids, int32_t T,
                 int64_t start_pos, int64_t *d_pos, float *d_h, float eps, void *d_ws, size_t ws_bytes,
                 uintptr_t stream, cudaEvent_t gate_wait = nullptr, const DevPos *dp = nullptr) {
    if (!hs || !layers) return ENGRAM_E_NULL;
    const DevPos dpos = dp ? *dp : DevPos{0, T, false};
    if (d_pos) start_pos = dpos.offset;
    int rc = check_hash(hs, d_ids, T, d_pos ? 0 : start_pos, d_ws);
    if (rc || T == 0) return rc;                  // T == 0: a valid no-op
    if (d_pos && !aligned(d_pos, 8)) return ENGRAM_E_ALIGN;
    if (!d_h) return ENGRAM_E_NULL;
    const engram_geom &g = hs->t->g;
    if (!(eps >= 0.0f)) return ENGRAM_E_INVALID;
    if (!aligned(d_h, 16) || !aligned(d_ws, 256)) return ENGRAM_E_ALIGN;
    const int L = g.n_layers, C = cols(g), hd = g.head_dim, K = C * hd, N = g.dim * (g.hc + 1);
    const int64_t M = (int64_t)hs->batch * T;
    bool all_q2k = K % 256 == 0;
    for (int l = 0; l < L; ++l) all_q2k = all_q2k && layers[l].wkv_q2k != nullptr;
    const bool use_q2k = all_q2k && M >= 1 && M <= kSmallT && K <= kGemvMaxK;
    for (int l = 0; l < L; ++l) {
        const engram_layer &ly = layers[l];
        if (!ly.table || !ly.qk) return ENGRAM_E_NULL;
        if (!ly.wkv && !use_q2k) return all_q2k && M >= 1 && M <= kSmallT ? ENGRAM_E_UNSUPPORTED : ENGRAM_E_NULL;
        if (ly.wkv_q2k && !aligned(ly.wkv_q2k, 16)) return ENGRAM_E_ALIGN;
        if (ly.wkv_tiled && !aligned(ly.wkv_tiled, 16)) return ENGRAM_E_ALIGN;
        if (ly.rows < 1) return ENGRAM_E_INVALID;
        if (ly.fmt == ENGRAM_FMT_FP8 || ly.fmt == ENGRAM_FMT_FP8_E8M0) {
            if (!ly.scales) return ENGRAM_E_NULL;
            if (!aligned(ly.table, 16) || (ly.fmt == ENGRAM_FMT_FP8 && !aligned(ly.scales, 4)))
                return ENGRAM_E_ALIGN;
        } else if (ly.fmt == ENGRAM_FMT_Q2K) {
            if (hd != 256) return ENGRAM_E_INVALID;      // one Q2_K block per 256-wide row
            if (!aligned(ly.table, 4)) return ENGRAM_E_ALIGN;
        } else {
            return ENGRAM_E_INVALID;
        }
        if (!aligned(ly.wkv, 16) || !aligned(ly.qk, 16)) return ENGRAM_E_ALIGN;
        if (!device_readable(ly.table) || (ly.scales && !device_readable(ly.scales))) return ENGRAM_E_INVALID;
    }
    if (M > (int64_t)1 << 24) return ENGRAM_E_UNSUPPORTED;
    if (ws_bytes < engram_workspace_bytes(&g, M)) return ENGRAM_E_WORKSPACE;
    if (M == 0) return ENGRAM_OK;
    int *err = err_ptr();
    if (!err) return ENGRAM_E_CUDA;
    cudaStream_t s = S(stream);
    size_t off[2 + 2 * kMaxLayers];
    engram_workspace_layout(&g, M, off);
    uint8_t *ws = static_cast<uint8_t *>(d_ws);
    int64_t *ids = reinterpret_cast<int64_t *>(ws + off[0]);

    // Small steps hash inside the projection kernel (each CTA hashes the ids
    // of its own layer); larger steps hash inside the row gather (one launch
    // for every layer); the rest (mixed table formats, odd head_dim) run the
    // hash kernel first.
    const bool small = gemv_fits((int)M, K);
    const bool fuse_hash = small && M * C <= kFusedHashMaxIds;
    HashRowsArgs hr{};
    hr.L = L;
    hr.M = M;
    for (int l = 0; l < L; ++l)
        hr.layer[l] = RowsArgs{static_cast<const uint8_t *>(layers[l].table), layers[l].scales, layers[l].rows,
                               hd, g.scale_block, ids + (int64_t)l * C, M, (int64_t)L * C, C,
                               reinterpret_cast<uint16_t *>(ws + off[1 + L + l]), err, layers[l].fmt};
    const bool hash_in_rows = !small && hash_rows_supported(hr);
    record(0, s);
    cudaError_t e = cudaSuccess;
    if (!fuse_hash && !hash_in_rows) {
        e = launch_hash(hash_args(hs, d_ids, T, start_pos, ids, d_pos, dpos.stable), s);
        if (e != cudaSuccess) return ENGRAM_E_CUDA;
    }
    record(1, s);

    GateArgs ga{};
    ga.h = d_h;
    ga.L = L;
    ga.M = (int32_t)M;
    ga.hc = g.hc;
    ga.D = g.dim;
    ga.eps = eps;
    ga.inv_sqrt_dim = powf((float)g.dim, -0.5f);
    ga.advance_pos = dpos.advance ? d_pos : nullptr;
    ga.advance_by = dpos.advance;
    for (int l = 0; l < L; ++l) {
        ga.kv[l] = reinterpret_cast<uint16_t *>(ws + off[1 + l]);
        ga.qk[l] = layers[l].qk;
    }

    if (small) {
        // Small step: one launch hashes, gathers every layer's rows into shared
        // memory and streams every layer's wkv; the gate follows it as a
        // programmatic dependent launch.
        GemvArgs a{};
        for (int l = 0; l < L; ++l) {
            a.layer[l].wkv = layers[l].wkv;
            a.layer[l].wkv_tiled = layers[l].wkv_tiled;
            a.layer[l].wkv_q2k = layers[l].wkv_q2k;
            a.layer[l].kv = reinterpret_cast<uint16_t *>(ws + off[1 + l]);
            a.layer[l].table = static_cast<const uint8_t *>(layers[l].table);
            a.layer[l].scales = layers[l].scales;
            a.layer[l].rows = layers[l].rows;
            a.layer[l].ids = ids + (int64_t)l * C;
            a.layer[l].fmt = layers[l].fmt;
        }
        a.L = L;
        a.T = (int32_t)M;
        a.K = K;
        a.N = N;
        a.hd = hd;
        a.blk = g.scale_block;
        a.C = C;
        a.id_stride = (int64_t)L * C;
        a.gather = 1;
        a.fuse_hash = fuse_hash ? 1 : 0;
        a.hash = hash_args(hs, d_ids, T, start_pos, ids, d_pos, dpos.stable);
        a.pdl = 1;
        a.sched = hs->sched;
        a.err = err;
        ga.pdl = 1;
        record(2, s);
        if ((use_q2k ? launch_gemv_q2k(a, s) : launch_gemv(a, s)) != cudaSuccess) return ENGRAM_E_CUDA;
        record(3, s);
    } else {
        if (hash_in_rows) {
            e = launch_hash_rows(hr, hash_args(hs, d_ids, T, start_pos, ids, d_pos, dpos.stable), s);
            if (e != cudaSuccess) return ENGRAM_E_CUDA;
        } else {
            for (int l = 0; l < L; ++l) {
                const RowsArgs &ra = hr.layer[l];
                e = layers[l].fmt == ENGRAM_FMT_Q2K ? launch_rows_q2k(ra, s) : launch_rows_fp8(ra, s);
                if (e != cudaSuccess) return ENGRAM_E_CUDA;
            }
        }
        record(2, s);
        const uint16_t *xs[kMaxLayers], *ws_[kMaxLayers];
        uint16_t *kvs[kMaxLayers];
        for (int l = 0; l < L; ++l) {
            xs[l] = reinterpret_cast<uint16_t *>(ws + off[1 + L + l]);
            ws_[l] = layers[l].wkv;
            kvs[l] = reinterpret_cast<uint16_t *>(ws + off[1 + l]);
        }
        if (gemm_tc_supported((int)M, N, K)) {
            // every layer's tiles in one persistent tensor-core launch
            // after the fused gather, launched early (see gemm_tc2.cu): 4096 tokens 1.221 ->
            // 1.215 ms a step, 512 tokens with Q2_K tables 0.1992 -> 0.1967 ms
            GemmTail tail{M >= 256 ? reinterpret_cast<float *>(ws + off[1 + 2 * L] - up256(kTailPartBytes))
                                   : nullptr};
            e = launch_gemm_tc(L, xs, ws_, kvs, (int)M, N, K, err, s, hash_in_rows, M >= 256 ? &tail : nullptr);

            if (e != cudaSuccess) return ENGRAM_E_CUDA;
        } else {
            for (int l = 0; l < L; ++l) {
                e = launch_gemm_simt(xs[l], ws_[l], kvs[l], (int)M, N, K, s);
                if (e != cudaSuccess) return ENGRAM_E_CUDA;
            }
        }
        record(3, s);
    }
    if (gate_wait && cudaStreamWaitEvent(s, gate_wait, 0) != cudaSuccess) return ENGRAM_E_CUDA;
    if (launch_gate(ga, s) != cudaSuccess) return ENGRAM_E_CUDA;
    record(4, s);
    return ENGRAM_OK;
}

}  // namespace

struct engram_graph {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

extern "C" {

int engram_forward(engram_hasher *hs, const engram_layer *layers, const int32_t *d_ids, int32_t T,
                   int64_t start_pos, float *d_h, float eps, void *d_ws, size_t ws_bytes, uintptr_t stream) {
    return forward_impl(hs, layers, d_ids, T, start_pos, nullptr, d_h, eps, d_ws, ws_bytes, stream);
}

int engram_forward_dpos(engram_hasher *hs, const engram_layer *layers, const int32_t *d_ids, int32_t T,
                        int64_t *d_start_pos, float *d_h, float eps, void *d_ws, size_t ws_bytes,
                        uintptr_t stream) {
    if (!d_start_pos) return ENGRAM_E_NULL;
    return forward_impl(hs, layers, d_ids, T, 0, d_start_pos, d_h, eps, d_ws, ws_bytes, stream);
}

int engram_graph_create_steps(engram_hasher *hs, const engram_layer *layers, const int32_t *d_ids, int32_t T,
                              int32_t steps, int64_t *d_start_pos, float *d_h, float eps, void *d_ws,
                              size_t ws_bytes, engram_graph **out) {
    if (!out) return ENGRAM_E_NULL;
    *out = nullptr;
    if (!hs || !layers || !d_start_pos || !d_ids || !d_h) return ENGRAM_E_NULL;
    if (T < 1 || steps < 1 || steps > 4096 || (int64_t)steps * T > hs->max_seq) return ENGRAM_E_INVALID;
    const engram_geom &geo = hs->t->g;
    const int64_t M = (int64_t)hs->batch * T;
    if (!err_ptr()) return ENGRAM_E_CUDA;            // looked up before the capture
    cudaStream_t cs;
    if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return ENGRAM_E_CUDA;
    const uintptr_t *prof = g_prof_events;
    g_prof_events = nullptr;                          // no profiling events inside the graph
    int rc = ENGRAM_OK;
    cudaGraph_t graph = nullptr;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        rc = ENGRAM_E_CUDA;
    } else {
        // Step k reads the position at *d_start_pos + k T; only the last step's
        // gate advances it (by steps T), so every step may hash ahead of the
        // previous step's gate, as eager calls from host positions do.
        for (int k = 0; k < steps && rc == ENGRAM_OK; ++k) {
            const DevPos dp{(int64_t)k * T, k == steps - 1 ? (int64_t)steps * T : 0, true};
            rc = forward_impl(hs, layers, d_ids + (int64_t)k * M, T, 0, d_start_pos,
                              d_h + (size_t)k * M * geo.hc * geo.dim, eps, d_ws, ws_bytes,
                              reinterpret_cast<uintptr_t>(cs), nullptr, &dp);
        }
        if (cudaStreamEndCapture(cs, &graph) != cudaSuccess && rc == ENGRAM_OK) rc = ENGRAM_E_CUDA;
    }
    g_prof_events = prof;
    cudaStreamDestroy(cs);
    if (rc != ENGRAM_OK) {
        if (graph) cudaGraphDestroy(graph);
        return rc;
    }
    engram_graph *g = new engram_graph();
    g->graph = graph;
    if (cudaGraphInstantiate(&g->exec, graph, 0) != cudaSuccess) {
        cudaGraphDestroy(graph);
        delete g;
        return ENGRAM_E_CUDA;
    }
    *out = g;
    return ENGRAM_OK;
}

int engram_graph_create(engram_hasher *hs, const engram_layer *layers, const int32_t *d_ids, int32_t T,
                        int64_t *d_start_pos, float *d_h, float eps, void *d_ws, size_t ws_bytes,
                        engram_graph **out) {
    return engram_graph_create_steps(hs, layers, d_ids, T, 1, d_start_pos, d_h, eps, d_ws, ws_bytes, out);
}

int engram_graph_launch(engram_graph *g, uintptr_t stream) {
    if (!g) return ENGRAM_E_NULL;
    return cuda_rc(cudaGraphLaunch(g->exec, S(stream)));
}

void engram_graph_destroy(engram_graph *g) {
    if (!g) return;
    cudaGraphExecDestroy(g->exec);
    cudaGraphDestroy(g->graph);
    delete g;
}

int engram_forward_host(engram_hasher *hs, const engram_layer *layers, const int32_t *h_ids, int32_t *d_ids,
                        int32_t T, int64_t start_pos, float *h_h, float *d_h, float eps, void *d_ws,
                        size_t ws_bytes, uintptr_t stream) {
    if (!hs || !h_ids || !d_ids || !h_h || !d_h) return ENGRAM_E_NULL;
    if (T < 0) return ENGRAM_E_INVALID;
    const engram_geom &g = hs->t->g;
    const size_t M = (size_t)hs->batch * T;
    const size_t hbytes = M * g.hc * g.dim * sizeof(float);
    cudaStream_t s = S(stream);
    if (start_pos < 0 || start_pos + T > hs->max_seq) return ENGRAM_E_CAPACITY;
    if (ws_bytes < engram_workspace_bytes(&g, (int64_t)M)) return ENGRAM_E_WORKSPACE;
    if (M == 0) return ENGRAM_OK;
    // Page-locked, device-mapped host buffers: the kernels read the ids and
    // update the highway in place over the CPU-GPU link -- no staging copies,
    // and consecutive steps keep their launch overlap.
    if (aligned(h_h, 16) && device_readable(h_ids) && device_readable(h_h))
        return forward_impl(hs, layers, h_ids, T, start_pos, nullptr, h_h, eps, d_ws, ws_bytes, stream);
    if (cudaMemcpyAsync(d_ids, h_ids, M * sizeof(int32_t), cudaMemcpyHostToDevice, s) != cudaSuccess)
        return ENGRAM_E_CUDA;
    // The highway upload goes on the hasher's auxiliary stream, after all
    // earlier work on the caller's stream (e.g. the previous read-back of
    // d_h), so it overlaps the projection; only the gate waits for it.
    if (cudaEventRecord(hs->ev_main, s) != cudaSuccess || cudaStreamWaitEvent(hs->aux, hs->ev_main, 0) != cudaSuccess ||
        cudaMemcpyAsync(d_h, h_h, hbytes, cudaMemcpyHostToDevice, hs->aux) != cudaSuccess ||
        cudaEventRecord(hs->ev_h, hs->aux) != cudaSuccess)
        return ENGRAM_E_CUDA;
    int rc = forward_impl(hs, layers, d_ids, T, start_pos, nullptr, d_h, eps, d_ws, ws_bytes, stream, hs->ev_h);
    if (rc) {
        cudaStreamWaitEvent(s, hs->ev_h, 0);         // leave no upload running past an error
        return rc;
    }
    return cuda_rc(cudaMemcpyAsync(h_h, d_h, hbytes, cudaMemcpyDeviceToHost, s));
}

}  // extern "C"
