// Shared definitions of the CUDA library (device and host side).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

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

__device__ inline float bf16_bits_to_float(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// Convert a CUDA error at enqueue time to a status code.
inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? D3D_OK : D3D_ERR_CUDA; }

inline bool ws_ok(const void *ws, size_t ws_bytes, size_t need)
{
    return ws != nullptr && (reinterpret_cast<uintptr_t>(ws) % kWsAlign) == 0 && ws_bytes >= need;
}

}  // namespace d3d
