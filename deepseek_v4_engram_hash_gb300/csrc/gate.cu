// gate.cu -- the engram gate (stage 4) for one or more layers on one highway.
//
// The gate of the CPU reference page "metrale_model_arch/deepseek_v41_ref/engram.rs"
// (module doc, item 4) on the FP32 highway of the GPU module page
// "spark_model/layers/engram_v41.rs" (module doc, item 4), per token t and
// stream c, with key = kv[t, c D : (c+1) D], value = kv[t, hc D : (hc+1) D]:
//   hh = sum h^2, kk = sum key^2, dot = sum (h (q k)) key
//   s  = dot * (1/sqrt(hh/D + eps) * 1/sqrt(kk/D + eps)) * D^-1/2
//   g  = copysign(sqrt(max(|s|, 1e-6)), s)
//   h += sigmoid(g) * value.
//
// One CTA per (token, stream) row of D values (128 or 256 threads).  The row stays in registers
// across the layers: layer l+1's norms and dot are taken on the highway that
// layer l just updated, so the highway is read and written once for all
// layers.  Reductions: per-thread f32 sums, a warp butterfly, then the
// per-warp partials summed in warp order -- a fixed order, reproducible.
#include "common.cuh"

namespace engram {

constexpr int kGateThreads = 256;

template <int TH>
__device__ __forceinline__ void block_sum3(float &a, float &b, float &c, float *red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        a += __shfl_xor_sync(0xFFFFFFFFu, a, off);
        b += __shfl_xor_sync(0xFFFFFFFFu, b, off);
        c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();                                  // red[] free from the last use
    if (lane == 0) {
        red[3 * warp + 0] = a;
        red[3 * warp + 1] = b;
        red[3 * warp + 2] = c;
    }
    __syncthreads();
    a = b = c = 0.0f;
#pragma unroll
    for (int w = 0; w < TH / 32; ++w) {
        a += red[3 * w + 0];
        b += red[3 * w + 1];
        c += red[3 * w + 2];
    }
}

// The per-layer operands of one thread: NV chunks of 4 key and value bf16
// and 4 q*k f32 values.
template <int NV>
struct GateChunk {
    uint2 kb[NV], vb[NV];
    float4 q[NV];
};

template <int NV, int TH>
__device__ __forceinline__ void load_qk(const GateArgs &a, int l, int c, GateChunk<NV> &g) {
    const int D4 = a.D >> 2;
    const float4 *qk = reinterpret_cast<const float4 *>(a.qk[l] + (size_t)c * a.D);
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int i = threadIdx.x + v * TH;
        g.q[v] = i < D4 ? __ldg(qk + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

template <int NV, int TH>
__device__ __forceinline__ void load_kv(const GateArgs &a, int l, int t, int c, GateChunk<NV> &g) {
    const int D4 = a.D >> 2;
    const size_t N = (size_t)a.D * (a.hc + 1);
    const uint16_t *kvt = a.kv[l] + (size_t)t * N;
    const uint2 *key = reinterpret_cast<const uint2 *>(kvt + (size_t)c * a.D);
    const uint2 *val = reinterpret_cast<const uint2 *>(kvt + (size_t)a.hc * a.D);
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int i = threadIdx.x + v * TH;
        g.kb[v] = i < D4 ? key[i] : make_uint2(0, 0);
        g.vb[v] = i < D4 ? val[i] : make_uint2(0, 0);
    }
}

// NV = float4 chunks per thread (D <= TH * 4 * NV, TH threads a CTA).  PIPE: the next
// layer's operands load while this layer reduces -- the latency choice for a
// handful of rows (one token).  Without it four CTAs share an SM -- the
// throughput choice for many rows, at 128 threads and 128 registers (32
// values a thread) up to D = 4096, at 256 threads and 64 registers beyond.
template <int NV, bool PIPE, int TH = kGateThreads>
__global__ void __launch_bounds__(TH, PIPE ? 1 : 4) gate_kernel(const __grid_constant__ GateArgs a) {
    constexpr bool kPipe = PIPE && NV <= 4;
    __shared__ float red[3 * TH / 32];
    const int row = blockIdx.x;                       // (t, c)
    const int t = row / a.hc, c = row % a.hc;
    const int D = a.D, D4 = D >> 2;
    float4 *hrow = reinterpret_cast<float4 *>(a.h + (size_t)row * D);
    // The highway and the first q*k do not depend on the projection: load
    // them before waiting for it.
    float4 h[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int i = threadIdx.x + v * TH;
        h[v] = i < D4 ? hrow[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    GateChunk<NV> cur, nxt;
    load_qk<NV, TH>(a, 0, c, cur);
    if (a.pdl) {
        griddep_wait();
        griddep_launch();
    }
    if (a.advance_pos && blockIdx.x == 0 && threadIdx.x == 0)
        *a.advance_pos += a.advance_by;     // every read of the position happened in the projection
    load_kv<NV, TH>(a, 0, t, c, cur);
    for (int l = 0; l < a.L; ++l) {
        if (kPipe && l + 1 < a.L) {
            load_qk<NV, TH>(a, l + 1, c, nxt);
            load_kv<NV, TH>(a, l + 1, t, c, nxt);
        }
        float hh = 0.f, kk = 0.f, dot = 0.f;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const float k0 = bf16_lo(cur.kb[v].x), k1 = bf16_hi(cur.kb[v].x);
            const float k2 = bf16_lo(cur.kb[v].y), k3 = bf16_hi(cur.kb[v].y);
            hh = fmaf(h[v].x, h[v].x, hh); hh = fmaf(h[v].y, h[v].y, hh);
            hh = fmaf(h[v].z, h[v].z, hh); hh = fmaf(h[v].w, h[v].w, hh);
            kk = fmaf(k0, k0, kk); kk = fmaf(k1, k1, kk);
            kk = fmaf(k2, k2, kk); kk = fmaf(k3, k3, kk);
            dot = fmaf(h[v].x * cur.q[v].x, k0, dot); dot = fmaf(h[v].y * cur.q[v].y, k1, dot);
            dot = fmaf(h[v].z * cur.q[v].z, k2, dot); dot = fmaf(h[v].w * cur.q[v].w, k3, dot);
        }
        block_sum3<TH>(hh, kk, dot, red);
        const float rstd = (1.0f / sqrtf(hh / (float)D + a.eps)) * (1.0f / sqrtf(kk / (float)D + a.eps));
        const float s = dot * rstd * a.inv_sqrt_dim;
        const float g = copysignf(sqrtf(fmaxf(fabsf(s), 1e-6f)), s);
        const float gate = 1.0f / (1.0f + expf(-g));
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            h[v].x = __fadd_rn(h[v].x, __fmul_rn(gate, bf16_lo(cur.vb[v].x)));
            h[v].y = __fadd_rn(h[v].y, __fmul_rn(gate, bf16_hi(cur.vb[v].x)));
            h[v].z = __fadd_rn(h[v].z, __fmul_rn(gate, bf16_lo(cur.vb[v].y)));
            h[v].w = __fadd_rn(h[v].w, __fmul_rn(gate, bf16_hi(cur.vb[v].y)));
        }
        if (l + 1 < a.L) {
            if (kPipe) {
                cur = nxt;
            } else {
                load_qk<NV, TH>(a, l + 1, c, cur);
                load_kv<NV, TH>(a, l + 1, t, c, cur);
            }
        }
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int i = threadIdx.x + v * TH;
        if (i < D4) hrow[i] = h[v];
    }
}

template <int NV, bool PIPE, int TH = kGateThreads>
static cudaError_t launch_nv(const GateArgs &a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.M * a.hc);
    cfg.blockDim = dim3(TH);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gate_kernel<NV, PIPE, TH>, a);
}

template <bool PIPE>
static cudaError_t launch_p(const GateArgs &a, cudaStream_t s) {
    const int per = kGateThreads * 4;
    if (a.D <= per) return launch_nv<1, PIPE>(a, s);
    if (a.D <= 2 * per) return launch_nv<2, PIPE>(a, s);
    if (a.D <= 4 * per) return launch_nv<4, PIPE>(a, s);
    if (a.D <= 8 * per) return launch_nv<8, false>(a, s);
    if (a.D <= 16 * per) return launch_nv<16, false>(a, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_gate(const GateArgs &a, cudaStream_t s) {
    if (a.M == 0) return cudaSuccess;
    // One CTA per (token, stream).  Few rows: 256 threads, the layers pipelined.
    // Many rows up to dim 4096: 128 threads, 8 float4 a thread in 128 registers,
    // four CTAs an SM (4096 tokens: 140.8 us against 148.7 with 256 threads at
    // 64 registers; 161 at 96 registers, which spill; 247 with 512 threads).
    if ((int64_t)a.M * a.hc <= 512) return launch_p<true>(a, s);
    constexpr int per = 128 * 4;
    if (a.D <= per) return launch_nv<1, false, 128>(a, s);
    if (a.D <= 2 * per) return launch_nv<2, false, 128>(a, s);
    if (a.D <= 4 * per) return launch_nv<4, false, 128>(a, s);
    if (a.D <= 8 * per) return launch_nv<8, false, 128>(a, s);
    return launch_p<false>(a, s);
}

}  // namespace engram
