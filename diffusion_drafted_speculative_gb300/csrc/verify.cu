// Speculative-sampling verification: host-side launch and the C entry points.
// The kernel (phases A-D) is in verify_body.cuh.
#include <math.h>

#include <mutex>

#include "greedy_body.cuh"
#include "verify_body.cuh"
#include "verify_slice.cuh"

namespace d3d {
namespace {

template <typename T, int NT>
int launch_verify_nt(const VArgs &a_in, int sm_limit, int flags, cudaStream_t stream)
{
    VArgs a = a_in;
    const VerifyLayout L = verify_layout(a.R, a.B, a.V, VCfg<NT>::kChunk);
    const long long nA = (long long)a.R * a.B * L.nch;
    if (nA > 0x7fffffffLL)
        return D3D_ERR_UNSUPPORTED;
    size_t dyn = verify_dyn_smem(a.B, L.nch);
    if (ring_fits<T, NT>(a)) {  // phase A through a shared-memory ring (one CTA per SM)
        const cudaError_t attr_err = set_max_dyn_smem<verify_kernel<T, NT>>((int)Ring<NT>::bytes(kRingSlots));
        if (attr_err == cudaSuccess) {
            a.ring = kRingSlots;
            if (dyn < Ring<NT>::bytes(kRingSlots))
                dyn = Ring<NT>::bytes(kRingSlots);
        } else {
            cudaGetLastError();
        }
    }
    // every CTA must be resident (CTAs wait on one another): at most the
    // occupancy limit (and the SM limit), and no more than there are phase-A items
    int dev = 0, nsm = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_kernel<T, NT>, NT, dyn) != cudaSuccess ||
        per_sm < 1)
        return D3D_ERR_CUDA;
    long long cap = (long long)nsm * per_sm;
    if (sm_limit > 0 && (long long)sm_limit * per_sm < cap)
        cap = (long long)sm_limit * per_sm;
    const unsigned grid = (unsigned)(nA < cap ? nA : cap);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    unsigned na = 1;
    if (flags & D3D_VERIFY_AFTER_INDEPENDENT) {  // may start while the previous kernel runs
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, verify_kernel<T, NT>, a);
    return cuda_status(e);
}

constexpr int kSliceSmemMax = 219 * 1024;  // dynamic shared memory of a slice CTA (227 KB per CTA less its static arrays)

// Slice width W (a multiple of kSliceGrain) and count nS when the request's
// rows split over the SMs the launch may use with every row of a slice
// resident in one CTA's shared memory, else false.  W is the smallest width
// that gives each request at most its share of the SMs.
inline int slice_width(int R, int V, int units)
{
    const int per = units / R;  // slices per request
    if (per < 1)
        return 0;
    const long long w = ((long long)V + per - 1) / per;
    return (int)((w + kSliceGrain - 1) / kSliceGrain * kSliceGrain);
}

// The workspace the slice launch can need: its finest slices (every unit a
// launch may hold) give the most records.
inline size_t slice_ws_bound(int R, int B, int V)
{
    const int W = slice_width(R, V, kSliceMaxUnits);
    return W > 0 ? verify_layout(R, B, V, W).total : 0;
}

template <typename T>
bool slice_plan(const VArgs &a, int sm_limit, size_t ws_bytes, int &W, int &nS, size_t &dyn)
{
    // rows and slices start on 16-byte boundaries (bulk copies)
    if ((size_t)a.V * sizeof(T) % 16 != 0 || (reinterpret_cast<uintptr_t>(a.target) & 15) != 0 ||
        (reinterpret_cast<uintptr_t>(a.draft) & 15) != 0)
        return false;
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    int units = (sm_limit > 0 && sm_limit < nsm) ? sm_limit : nsm;
    if (units > kSliceMaxUnits)
        units = kSliceMaxUnits;
    W = slice_width(a.R, a.V, units);
    if (W <= 0)
        return false;
    nS = (a.V + W - 1) / W;
    dyn = SliceLayout<T>(a.B, W, nS).total;
    if (dyn > (size_t)kSliceSmemMax || verify_layout(a.R, a.B, a.V, W).total > ws_bytes)
        return false;
    return set_max_dyn_smem<verify_slice_kernel<T>>(kSliceSmemMax) == cudaSuccess;
}

template <typename T>
int launch_verify_slice(const VArgs &a, int W, int nS, size_t dyn, int flags, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.R * nS));
    cfg.blockDim = dim3(kSliceThreads);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;  // the CTAs of a request wait on one another
    attr[0].val.cooperative = 1;
    unsigned na = 1;
    if (flags & D3D_VERIFY_AFTER_INDEPENDENT) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cuda_status(cudaLaunchKernelEx(&cfg, verify_slice_kernel<T>, a, W, nS));
}

// The slice launch when the call's requests split over the SMs with their
// slices resident in shared memory; otherwise the chunked kernel: with an SM
// limit its CTAs are 512 threads, one per SM (the register file holds one),
// so a launch beside another kernel takes at most sm_limit SMs.
template <typename T>
int launch_verify(const VArgs &a, int sm_limit, int flags, cudaStream_t stream, size_t ws_bytes)
{
    int W = 0, nS = 0;
    size_t dyn = 0;
    if (slice_plan<T>(a, sm_limit, ws_bytes, W, nS, dyn))
        return launch_verify_slice<T>(a, W, nS, dyn, flags, stream);
    cudaGetLastError();
    if (sm_limit > 0)
        return launch_verify_nt<T, kNTLimited>(a, sm_limit, flags, stream);
    return launch_verify_nt<T, kNTDevice>(a, 0, flags, stream);
}

}  // namespace
}  // namespace d3d

extern "C" {

size_t d3d_spec_verify_workspace_size(int R, int B, int V)
{
    if (R < 0 || B < 2 || V < 1 || B > d3d::kMaxB || V > d3d::kMaxChunks * d3d::kVChunkMin)
        return 0;
    // the smaller chunk has the most records: the workspace fits both chunked
    // launches; the slice launch needs at most slice_ws_bound
    const size_t chunked = d3d::verify_layout(R, B, V, d3d::kVChunkMin).total;
    const size_t sliced = d3d::slice_ws_bound(R, B, V);
    return chunked > sliced ? chunked : sliced;
}

int d3d_spec_verify_slice_ctas(int R, int B, int V, int logits_dtype, float temperature, int sm_limit,
                               size_t ws_bytes)
{
    if (R < 0 || B < 2 || B > d3d::kMaxB || V < 1 || V > d3d::kMaxChunks * d3d::kVChunkMin || sm_limit < 0 ||
        !(temperature >= 0.f) || (logits_dtype != D3D_DTYPE_BF16 && logits_dtype != D3D_DTYPE_F32))
        return D3D_ERR_INVALID_ARG;
    if (R == 0 || temperature == 0.f)
        return 0;  // nothing to launch, or the greedy launch
    d3d::VArgs a{};
    a.R = R, a.B = B, a.V = V;
    static __align__(16) unsigned char probe[16];  // stands for 16-byte aligned rows
    a.target = a.draft = probe;
    int W = 0, nS = 0;
    size_t dyn = 0;
    const bool sliced = logits_dtype == D3D_DTYPE_BF16 ? d3d::slice_plan<uint16_t>(a, sm_limit, ws_bytes, W, nS, dyn)
                                                       : d3d::slice_plan<float>(a, sm_limit, ws_bytes, W, nS, dyn);
    cudaGetLastError();
    return sliced ? R * nS : 0;
}

int d3d_spec_verify(const void *target_logits, const void *draft_logits, int logits_dtype,
                    const int32_t *draft_tokens, const float *u_accept, const float *u_sample, int R, int B,
                    int V, float temperature, int32_t *accept_len, int32_t *out_tokens, int32_t *num_tokens,
                    float *alpha, float *p_draft, float *q_draft, float *awl_weight, const int32_t *heads,
                    const int32_t *head_len, int M, int32_t *branch, void *ws, size_t ws_bytes, int sm_limit,
                    int flags, cudaStream_t stream)
{
    if (sm_limit < 0 || (flags & ~D3D_VERIFY_AFTER_INDEPENDENT) != 0)
        return D3D_ERR_INVALID_ARG;
    d3d::VArgs a;
    const int rc = d3d::verify_prepare(target_logits, draft_logits, logits_dtype, draft_tokens, u_accept, u_sample,
                                       R, B, V, temperature, accept_len, out_tokens, num_tokens, alpha, p_draft,
                                       q_draft, awl_weight, heads, head_len, M, branch, a);
    if (rc != D3D_OK)
        return rc == 1 ? D3D_OK : rc;
    if (!d3d::ws_ok(ws, ws_bytes, d3d::verify_layout(R, B, V, d3d::kVChunkMin).total))
        return D3D_ERR_WORKSPACE;
    a.ws = static_cast<unsigned char *>(ws);
    if (temperature == 0.f)
        return logits_dtype == D3D_DTYPE_BF16 ? d3d::launch_greedy<uint16_t>(a, sm_limit, flags, stream)
                                              : d3d::launch_greedy<float>(a, sm_limit, flags, stream);
    if (logits_dtype == D3D_DTYPE_BF16)
        return d3d::launch_verify<uint16_t>(a, sm_limit, flags, stream, ws_bytes);
    return d3d::launch_verify<float>(a, sm_limit, flags, stream, ws_bytes);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Verification without a caller workspace.
//
// For callers that cannot allocate device memory, the scratch the
// verification kernel needs lives in one fixed, file-scope device array.
// Every device that loads this library holds it until the process exits.
// ---------------------------------------------------------------------------
namespace d3d {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;  // 2 MiB
constexpr int kNoAllocMaxDevices = 64;

std::mutex g_noalloc_mu;
void *g_noalloc_addr[kNoAllocMaxDevices];

}  // namespace
}  // namespace d3d

static __device__ __align__(256) unsigned char d3d_noalloc_verify_scratch[d3d::kNoAllocScratchBytes];

namespace d3d {
namespace {

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current, and cached.
int noalloc_scratch(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return D3D_ERR_CUDA;
    }
    if (dev < 0 || dev >= kNoAllocMaxDevices)
        return D3D_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, d3d_noalloc_verify_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return D3D_ERR_CUDA;
        }
        g_noalloc_addr[dev] = ptr;
    }
    *out = g_noalloc_addr[dev];
    return D3D_OK;
}

}  // namespace
}  // namespace d3d

extern "C" int d3d_spec_verify_noalloc(const void *target_logits, const void *draft_logits, int logits_dtype,
                                       const int32_t *draft_tokens, const float *u_accept, const float *u_sample,
                                       int R, int B, int V, float temperature, int32_t *accept_len,
                                       int32_t *out_tokens, int32_t *num_tokens, float *alpha, float *p_draft,
                                       float *q_draft, cudaStream_t stream)
{
    d3d::VArgs a;
    const int rc = d3d::verify_prepare(target_logits, draft_logits, logits_dtype, draft_tokens, u_accept, u_sample,
                                       R, B, V, temperature, accept_len, out_tokens, num_tokens, alpha, p_draft,
                                       q_draft, nullptr, nullptr, nullptr, 0, nullptr, a);
    if (rc != D3D_OK)
        return rc == 1 ? D3D_OK : rc;
    const d3d::VerifyLayout L = d3d::verify_layout(R, B, V, d3d::kVChunkMin);
    if (L.total > d3d::kNoAllocScratchBytes)
        return D3D_ERR_UNSUPPORTED;  // needs more scratch than the fixed array holds
    void *scratch = nullptr;
    const int rs = d3d::noalloc_scratch(&scratch);
    if (rs != D3D_OK)
        return rs;
    // the array keeps the previous call's contents: zero the status word and
    // the per-request counters, which must start at zero
    if (cudaMemsetAsync(scratch, 0, L.rec, stream) != cudaSuccess)
        return D3D_ERR_CUDA;
    a.ws = static_cast<unsigned char *>(scratch);
    if (temperature == 0.f)
        return logits_dtype == D3D_DTYPE_BF16 ? d3d::launch_greedy<uint16_t>(a, 0, 0, stream)
                                              : d3d::launch_greedy<float>(a, 0, 0, stream);
    if (logits_dtype == D3D_DTYPE_BF16)
        return d3d::launch_verify<uint16_t>(a, 0, 0, stream, d3d::kNoAllocScratchBytes);
    return d3d::launch_verify<float>(a, 0, 0, stream, d3d::kNoAllocScratchBytes);
}
