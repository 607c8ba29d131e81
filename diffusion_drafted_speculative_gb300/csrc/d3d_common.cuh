// Shared definitions of the CUDA library (device and host side).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "d3d.h"

namespace d3d {

// Every workspace starts with this header; the rest is per-entry-point.
struct WsHeader {
    int32_t status;  // D3D_OK or the first device-side error recorded
    int32_t pad[63];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

constexpr size_t kWsAlign = 256;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Record the first device-side error in the workspace status word.
__device__ inline void record_status(int32_t *status, int32_t code)
{
    atomicCAS(reinterpret_cast<int *>(status), D3D_OK, code);
}

// Internal index checks of the debug build (compiled with D3D_DEBUG_CHECKS):
// a failed check records D3D_ERR_INTERNAL in the status word and returns
// false, and the caller skips the access; it never traps.  In the normal
// build the check is compiled out and returns true.
#ifdef D3D_DEBUG_CHECKS
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif
__device__ __forceinline__ bool dbg_ok(bool cond, int32_t *status)
{
    if (kDebugChecks && !cond) {
        record_status(status, D3D_ERR_INTERNAL);
        return false;
    }
    return true;
}

__device__ inline float bf16_bits_to_float(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// One logit as float (f32, or bf16 bits: exact), read through the read-only path.
__device__ inline float load_logit(const float *p, long long i) { return __ldg(p + i); }
__device__ inline float load_logit(const uint16_t *p, long long i) { return bf16_bits_to_float(__ldg(p + i)); }

// 8 consecutive logits from a 16-byte aligned address.
__device__ inline void load_logits8(const float *p, float (&x)[8])
{
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p)), b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
}
__device__ inline void load_logits8(const uint16_t *p, float (&x)[8])
{
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(wv[e] << 16);
        x[2 * e + 1] = __uint_as_float(wv[e] & 0xffff0000u);
    }
}

// Failure-injection mode of the host hook d3d_debug_inject_fault (one value
// for the whole library; 0 = normal operation).  Read at launch time and
// passed to the kernels as an argument.
inline int &fault_mode()
{
    static int mode = 0;
    return mode;
}

// Raise kernel K's dynamic shared-memory limit to `bytes` on the current
// device, once per device (a function attribute belongs to the device it
// was set on); thread-safe.  Returns the result of the (first) call.
template <auto K> inline cudaError_t set_max_dyn_smem(int bytes)
{
    constexpr int kDev = 64;
    static std::mutex mu;
    static bool done[kDev];
    static cudaError_t err[kDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return cudaErrorInvalidDevice;
    }
    if (dev < 0 || dev >= kDev)
        return cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
        err[dev] = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        done[dev] = true;
    }
    return err[dev];
}

// Convert a CUDA error at enqueue time to a status code.
inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? D3D_OK : D3D_ERR_CUDA; }

inline bool ws_ok(const void *ws, size_t ws_bytes, size_t need)
{
    return ws != nullptr && (reinterpret_cast<uintptr_t>(ws) % kWsAlign) == 0 && ws_bytes >= need;
}

}  // namespace d3d
