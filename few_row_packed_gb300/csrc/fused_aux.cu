// fused_aux.cu -- test export of the fused head's activation rotation (the
// prologue device functions of the few-row kernel -- sign flip and blockwise
// FWHT-128 on the tensor cores -- run on their own, so their output can be
// compared element by element), and the module-owned scratch of
// lbv_verify_fused_noalloc.
#include <mutex>

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
    rotate_x<XT>(smem_u32(xs), RS, have / 128, threadIdx.x >> 5, 8, threadIdx.x & 31);
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

// ---------------------------------------------------------------------------
// Scratch of lbv_verify_fused_noalloc: the argmax keys of up to 8 rows and the
// count of finished CTAs (the layout of lbv_verify_fused's workspace), in the
// module's own device memory, zero at load and left zero by every call.

namespace {

constexpr size_t kNoAllocScratch = 256;          // bytes; the workspace needs 128
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratch];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices];                // symbol address per device, once
bool g_scratch_cleared[kMaxDevices];

}  // namespace

namespace lbv {

size_t noalloc_scratch_bytes()
{
    return kNoAllocScratch;
}

// The scratch of the current device: its symbol address, looked up once per
// device (a cudaDeviceReset invalidates it for the rest of the process).
// *needs_clear stays true until noalloc_scratch_cleared() records that a
// clear of the device's scratch was enqueued, so a failed clear is retried on
// the next call.
cudaError_t noalloc_scratch(void** out, bool* needs_clear)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    *needs_clear = !g_scratch_cleared[dev];
    return cudaSuccess;
}

// Records that the clear of the current device's scratch was enqueued.
void noalloc_scratch_cleared()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    g_scratch_cleared[dev] = true;
}

}  // namespace lbv
