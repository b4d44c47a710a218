// synth.cu -- CUDA twin of the seeded input generator (synth.py).
//
// Input generation only, built into its own library (libengram_synth.so);
// no part of the engram method is computed here.  Element i of a stream with
// key k is SplitMix64's mix of k + (i + 1) * 0x9E3779B97F4A7C15 (Steele, Lea
// & Flood, OOPSLA 2014).  Normals are the centred sum of the four 16-bit
// fields times one f32 constant; fp8, bf16 and fp16 come from CUDA's own
// round-to-nearest-even conversions.  Every step matches the numpy twin bit
// for bit.
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

__device__ __forceinline__ float normal(uint64_t z, float c) {
    const int64_t s = (int64_t)(z & 0xFFFF) + (int64_t)((z >> 16) & 0xFFFF) +
                      (int64_t)((z >> 32) & 0xFFFF) + (int64_t)(z >> 48);
    return __fmul_rn((float)(s - 2 * 65535), c);
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
