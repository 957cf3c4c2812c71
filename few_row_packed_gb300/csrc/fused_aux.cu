// fused_aux.cu -- test export of the fused head's activation rotation: the
// prologue device functions of the few-row kernel (sign flip and blockwise
// FWHT-128 on the tensor cores) run on their own, so their output can be
// compared element by element.
#include "verify_kernel.cuh"

namespace lbv {

// Each CTA (8 warps) stages 8 blocks of 128 elements of rows 0..7 in the
// verify kernel's shared-memory row layout (rows >= M zero), applies the same
// sign flip and rotation, and writes rows < M back.
template <int XT>
__global__ void __launch_bounds__(256) lbv_fused_rotation_kernel(const uint16_t* X, uint16_t* Xr,
                                                                 int M, int K,
                                                                 const uint32_t* signs)
{
    constexpr int BPC = 8;                               // blocks per CTA
    constexpr int RS = BPC * 256 + 16;                   // RS / 4 = 4 mod 8
    __shared__ __align__(16) unsigned char xs[8 * RS];
    const int kb = blockIdx.x * BPC * 128;
    const int have = min(BPC * 128, K - kb);
    for (int i = threadIdx.x; i < 8 * have; i += 256) {
        const int m = i / have, k = i - m * have;
        reinterpret_cast<uint16_t*>(xs + m * RS)[k] =
            m < M ? X[(size_t)m * K + kb + k] : (uint16_t)0;
    }
    __syncthreads();
    if (signs) {
        flip_signs(signs, xs, RS, M, kb, have, threadIdx.x, 256);
        __syncthreads();
    }
    rotate_x<XT>(smem_u32(xs), xs, RS, have / 128, threadIdx.x >> 5, 8, threadIdx.x & 31);
    __syncthreads();
    for (int i = threadIdx.x; i < M * have; i += 256) {
        const int m = i / have, k = i - m * have;
        Xr[(size_t)m * K + kb + k] = reinterpret_cast<const uint16_t*>(xs + m * RS)[k];
    }
}

cudaError_t launch_fused_rotation(const void* X, void* Xr, int M, int K, lbv_dtype dt,
                                  const uint32_t* signs, cudaStream_t st)
{
    const dim3 grid((unsigned)((K / 128 + 7) / 8));
    if (dt == LBV_F16)
        lbv_fused_rotation_kernel<LBV_F16><<<grid, 256, 0, st>>>(
            static_cast<const uint16_t*>(X), static_cast<uint16_t*>(Xr), M, K, signs);
    else
        lbv_fused_rotation_kernel<LBV_BF16><<<grid, 256, 0, st>>>(
            static_cast<const uint16_t*>(X), static_cast<uint16_t*>(Xr), M, K, signs);
    return cudaGetLastError();
}

}  // namespace lbv
