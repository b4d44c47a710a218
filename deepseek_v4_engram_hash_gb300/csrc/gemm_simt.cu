// gemm_simt.cu -- plain shared-memory-tiled CUDA-core GEMM for the wkv
// projection, kv [M, N] = bf16_rne(x [M, K] . wkv [N, K]^T), f32 accumulation
// (page "metrale_model_arch/deepseek_v41_ref/engram.rs", module doc, item 3).
//
// 128 x 128 output tile per CTA, K in steps of 32, 256 threads with an 8 x 8
// register tile each.  This is the simple correct path for shapes the
// tensor-core GEMM does not take.
#include "common.cuh"

namespace engram {

constexpr int kSM = 128, kSN = 128, kSK = 32;

__global__ void __launch_bounds__(256) gemm_simt_kernel(const uint16_t *__restrict__ x,
                                                        const uint16_t *__restrict__ w,
                                                        uint16_t *__restrict__ kv, int M, int N,
                                                        int K) {
    __shared__ float As[kSK][kSM + 4];
    __shared__ float Bs[kSK][kSN + 4];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int m0 = blockIdx.y * kSM, n0 = blockIdx.x * kSN;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    for (int k0 = 0; k0 < K; k0 += kSK) {
        // 128 rows x 32 k = 512 chunks of 8 bf16 per operand; 2 per thread.
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int q = tid + 256 * r;
            const int row = q >> 2, kc = (q & 3) * 8;
            uint4 va = make_uint4(0, 0, 0, 0), vb = make_uint4(0, 0, 0, 0);
            if (m0 + row < M) va = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(m0 + row) * K + k0 + kc));
            if (n0 + row < N) vb = __ldg(reinterpret_cast<const uint4 *>(w + (size_t)(n0 + row) * K + k0 + kc));
            const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                As[kc + 2 * e][row] = bf16_lo(wa[e]);
                As[kc + 2 * e + 1][row] = bf16_hi(wa[e]);
                Bs[kc + 2 * e][row] = bf16_lo(wb[e]);
                Bs[kc + 2 * e + 1][row] = bf16_hi(wb[e]);
            }
        }
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < kSK; ++k) {
            float a[8], b[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = As[k][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 8; ++j) b[j] = Bs[k][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int m = m0 + ty + 16 * i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int n = n0 + tx + 16 * j;
            if (n < N) kv[(size_t)m * N + n] = (uint16_t)f32_to_bf16_bits(acc[i][j]);
        }
    }
}

cudaError_t launch_gemm_simt(const uint16_t *x, const uint16_t *wkv, uint16_t *kv, int M, int N,
                             int K, cudaStream_t s) {
    if (M == 0) return cudaSuccess;
    dim3 grid((N + kSN - 1) / kSN, (M + kSM - 1) / kSM);
    gemm_simt_kernel<<<grid, 256, 0, s>>>(x, wkv, kv, M, N, K);
    return cudaGetLastError();
}

}  // namespace engram
