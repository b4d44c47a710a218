// gemm.cu -- dispatch of the projection GEMM: the tcgen05 tensor-core kernels
// for every shape they take (K % 64 == 0, N % 8 == 0) -- CTA pairs from 256
// tokens (gemm_tc2.cu), one CTA below (gemm_tc.cu) -- and the CUDA-core
// kernel (gemm_simt.cu) otherwise.
#include "common.cuh"

namespace engram {

cudaError_t launch_gemm(const uint16_t *x, const uint16_t *wkv, uint16_t *kv, int M, int N, int K,
                        int *err, cudaStream_t s) {
    if (gemm_tc_supported(M, N, K)) return launch_gemm_tc(1, &x, &wkv, &kv, M, N, K, err, s);
    return launch_gemm_simt(x, wkv, kv, M, N, K, s);
}

}  // namespace engram
