// synth.cu -- CUDA twin of the seeded input generator (synth.py).
//
// Input generation only, built into its own library (libengram_synth.so);
// no part of the engram method is computed here.  Element i of a stream with
// key k is SplitMix64's mix of k + (i + 1) * 0x9E3779B97F4A7C15 (Steele, Lea
// & Flood, OOPSLA 2014).  Normals are N(0, 1) by the Box-Muller transform of
// one 64-bit output, evaluated in float64 from the series of ln and cos/sin
// with the same fixed sequence of correctly rounded operations (__dadd_rn,
// __dmul_rn, __ddiv_rn, __dsqrt_rn: nothing fused) and the same constants as
// the numpy twin, rounded to f32 and times one f32 sigma; fp8, bf16 and fp16
// come from CUDA's own round-to-nearest-even conversions.  Every step matches
// the numpy twin bit for bit.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t sm64(uint64_t key, uint64_t i) {
    uint64_t z = (i + 1ull) * 0x9E3779B97F4A7C15ull + key;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// ln 2, pi / 2, sqrt(1/2) and the series coefficients 1 / (2k + 1), (-1)^k /
// (2k)!, (-1)^k / (2k + 1)!: the doubles nearest the exact values.
__constant__ double kAtanh[11] = {
    0x1.0000000000000p+0, 0x1.5555555555555p-2, 0x1.999999999999ap-3, 0x1.2492492492492p-3,
    0x1.c71c71c71c71cp-4, 0x1.745d1745d1746p-4, 0x1.3b13b13b13b14p-4, 0x1.1111111111111p-4,
    0x1.e1e1e1e1e1e1ep-5, 0x1.af286bca1af28p-5, 0x1.8618618618618p-5};
__constant__ double kCos[10] = {
    0x1.0000000000000p+0, -0x1.0000000000000p-1, 0x1.5555555555555p-5, -0x1.6c16c16c16c17p-10,
    0x1.a01a01a01a01ap-16, -0x1.27e4fb7789f5cp-22, 0x1.1eed8eff8d898p-29, -0x1.93974a8c07c9dp-37,
    0x1.ae7f3e733b81fp-45, -0x1.6827863b97d97p-53};
__constant__ double kSin[10] = {
    0x1.0000000000000p+0, -0x1.5555555555555p-3, 0x1.1111111111111p-7, -0x1.a01a01a01a01ap-13,
    0x1.71de3a556c734p-19, -0x1.ae64567f544e4p-26, 0x1.6124613a86d09p-33, -0x1.ae7f3e733b81fp-41,
    0x1.952c77030ad4ap-49, -0x1.2f49b46814157p-57};
constexpr double kLn2 = 0x1.62e42fefa39efp-1, kPi2 = 0x1.921fb54442d18p+0, kSqrtHalf = 0x1.6a09e667f3bcdp-1;

// N(0, 1) from one SplitMix64 output: sqrt(-2 ln u1) cos(2 pi u2), u1 = (a + 1)
// 2^-32, u2 = b 2^-32 (a, b the high and low 32 bits).
__device__ double std_normal(uint64_t z) {
    int e = 0;
    double m0 = frexp((double)((z >> 32) + 1ull), &e);            // exact
    if (m0 < kSqrtHalf) {
        m0 = __dmul_rn(m0, 2.0);
        e -= 1;
    }
    const double s = __ddiv_rn(__dadd_rn(m0, -1.0), __dadd_rn(m0, 1.0));
    const double s2 = __dmul_rn(s, s);
    double p = kAtanh[10];
    for (int k = 9; k >= 0; --k) p = __dadd_rn(__dmul_rn(p, s2), kAtanh[k]);
    p = __dmul_rn(__dmul_rn(p, s), 2.0);                            // ln m0
    double l = __dmul_rn(__dadd_rn((double)e, -32.0), kLn2);
    l = __dmul_rn(__dadd_rn(l, p), -2.0);                          // -2 ln u1
    const double r = __dsqrt_rn(l);
    const double w = __dmul_rn((double)(uint32_t)z, 0x1p-30);       // 4 u2, exact
    const double q = floor(__dadd_rn(w, 0.5));
    const double x = __dmul_rn(__dadd_rn(w, -q), kPi2);
    const double x2 = __dmul_rn(x, x);
    // only the series the quadrant needs (the same operations as either of the twin's)
    const int qi = (int)q;
    const double *coef = (qi & 1) ? kSin : kCos;
    double v = coef[9];
    for (int k = 8; k >= 0; --k) v = __dadd_rn(__dmul_rn(v, x2), coef[k]);
    if (qi & 1) v = __dmul_rn(v, x);
    if (qi == 1 || qi == 2) v = -v;
    return __dmul_rn(r, v);
}

__device__ __forceinline__ float normal(uint64_t z, float c) {
    return __fmul_rn(__double2float_rn(std_normal(z)), c);
}

__global__ void fp8_table_kernel(uint64_t kt, uint64_t ks, int64_t R, int hd, int nb, float c,
                                 uint8_t *codes, float *scales) {
    const int64_t n = R * hd, stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        float x = normal(sm64(kt, (uint64_t)i), c);
        x = fminf(fmaxf(x, -448.0f), 448.0f);
        codes[i] = (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
        if (i < R * nb) {
            const int k = (int)(sm64(ks, (uint64_t)i) % 7ull) - 4;
            scales[i] = __uint_as_float((uint32_t)(k + 127) << 23);
        }
    }
}

__global__ void q2k_table_kernel(uint64_t key, int64_t R, float step, float lo, uint8_t *out) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < R; r += stride) {
        uint32_t *dst = reinterpret_cast<uint32_t *>(out + r * 84);
        for (int j = 0; j < 10; ++j) {
            const uint64_t z = sm64(key, (uint64_t)r * 12 + j);
            dst[2 * j] = (uint32_t)z;
            dst[2 * j + 1] = (uint32_t)(z >> 32);
        }
        uint16_t h[2];
        for (int j = 0; j < 2; ++j) {
            const uint64_t z = sm64(key, (uint64_t)r * 12 + 10 + j);
            const float u = (float)(uint32_t)(z >> 40);
            h[j] = __half_as_ushort(__float2half_rn(__fadd_rn(__fmul_rn(u, step), lo)));
        }
        dst[20] = (uint32_t)h[0] | ((uint32_t)h[1] << 16);
    }
}

__global__ void bf16_normal_kernel(uint64_t key, int64_t n, float c, uint16_t *out) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        out[i] = __bfloat16_as_ushort(__float2bfloat16_rn(normal(sm64(key, (uint64_t)i), c)));
}

__global__ void f32_normal_kernel(uint64_t key, int64_t first, int64_t n, float c, float *out) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        out[i] = normal(sm64(key, (uint64_t)(first + i)), c);
}

unsigned grid(int64_t n) {
    int64_t b = (n + 255) / 256;
    return (unsigned)(b > 152 * 32 ? 152 * 32 : (b < 1 ? 1 : b));
}

}  // namespace

extern "C" {

int synth_fp8_table(uint64_t key_table, uint64_t key_scales, int64_t R, int hd, int blk, float c,
                    void *codes, void *scales, void *stream) {
    fp8_table_kernel<<<grid(R * hd), 256, 0, (cudaStream_t)stream>>>(
        key_table, key_scales, R, hd, hd / blk, c, (uint8_t *)codes, (float *)scales);
    return (int)cudaGetLastError();
}

int synth_q2k_table(uint64_t key, int64_t R, float step, float lo, void *out, void *stream) {
    q2k_table_kernel<<<grid(R), 256, 0, (cudaStream_t)stream>>>(key, R, step, lo, (uint8_t *)out);
    return (int)cudaGetLastError();
}

int synth_bf16_normal(uint64_t key, int64_t n, float c, void *out, void *stream) {
    bf16_normal_kernel<<<grid(n), 256, 0, (cudaStream_t)stream>>>(key, n, c, (uint16_t *)out);
    return (int)cudaGetLastError();
}

int synth_f32_normal(uint64_t key, int64_t first, int64_t n, float c, void *out, void *stream) {
    f32_normal_kernel<<<grid(n), 256, 0, (cudaStream_t)stream>>>(key, first, n, c, (float *)out);
    return (int)cudaGetLastError();
}

}  // extern "C"
