// Host runtime: status word, workspace cache, SM count, tensor-map encoding,
// error strings. No kernels live here.

#include <cudaTypedefs.h>

#include <map>
#include <atomic>
#include <mutex>
#include <utility>
#include <vector>

#include "gqa_attn.h"
#include "ptx.cuh"
#include "runtime.cuh"

namespace gqa {

// The device status word lives in this module's own device memory, one copy
// per GPU, so reading or clearing it never allocates. Kernels receive its
// device address as a parameter (host code only has a host-side stand-in for
// the symbol, looked up per device below).
static __device__ unsigned g_status_word;

namespace {

constexpr int kMaxDevices = 64;
std::atomic<unsigned*> g_status[kMaxDevices];  // device -> address of g_status_word
std::atomic<int> g_sms[kMaxDevices];            // device -> SM count (0: not read yet)
std::mutex g_mu;

struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
    // Buffers replaced by a larger one. They are never freed: a CUDA graph
    // captured earlier on this stream may still use one. Each growth at least
    // doubles the size, so together they stay below the current buffer.
    std::vector<void*> retired;
};
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

}  // namespace

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

bool device_attrs_pending(const std::atomic<uint64_t>& done, int dev) {
    return dev < 0 || dev >= 64 || !(done.load(std::memory_order_acquire) & (uint64_t(1) << dev));
}

void device_attrs_mark(std::atomic<uint64_t>& done, int dev) {
    if (dev >= 0 && dev < 64) done.fetch_or(uint64_t(1) << dev, std::memory_order_release);
}

unsigned* status_word() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    unsigned* p = g_status[dev].load(std::memory_order_acquire);
    if (p) return p;
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_status_word) != cudaSuccess) return nullptr;
    p = static_cast<unsigned*>(a);
    g_status[dev].store(p, std::memory_order_release);
    return p;
}

int num_sms() {
    const int dev = current_device();
    if (dev < 0) return -1;
    if (dev < kMaxDevices) {
        const int n = g_sms[dev].load(std::memory_order_relaxed);
        if (n > 0) return n;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (dev < kMaxDevices) g_sms[dev].store(n, std::memory_order_relaxed);
    return n;
}

void* stream_workspace(cudaStream_t stream, size_t bytes) {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    Workspace& w = g_ws[{dev, stream}];
    if (w.bytes >= bytes && w.ptr) return w.ptr;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
        return nullptr;
    // Grow by at least 2x so a sequence of growing calls allocates O(log) times.
    size_t want = bytes > 2 * w.bytes ? bytes : 2 * w.bytes;
    void* p = nullptr;
    if (cudaMallocAsync(&p, want, stream) != cudaSuccess) return nullptr;
    if (w.ptr) w.retired.push_back(w.ptr);
    w.ptr = p;
    w.bytes = want;
    return p;
}

static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                             cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return nullptr;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    return g_encode;
}

cudaError_t encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t elem_bytes,
                        uint32_t rank, const void* base, const uint64_t* dims, const uint32_t* box,
                        CUtensorMapSwizzle swizzle) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc || rank < 1 || rank > 5) return cudaErrorSymbolNotFound;
    cuuint64_t d[5], strides[4];
    cuuint32_t bx[5], estr[5];
    uint64_t stride = elem_bytes;
    for (uint32_t i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        estr[i] = 1;
        if (i > 0) strides[i - 1] = stride;
        stride *= dims[i];
    }
    CUresult r = enc(map, dtype, rank, const_cast<void*>(base), d, strides, bx, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                                uint64_t outer, uint32_t box_inner, uint32_t box_rows,
                                CUtensorMapSwizzle swizzle) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return cudaErrorSymbolNotFound;
    cuuint64_t dims[3] = {inner, rows, outer};
    cuuint64_t strides[2] = {inner * 2, inner * rows * 2};  // bytes, dims 1 and 2
    cuuint32_t box[3] = {box_inner, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Test hook (gqa_attn_debug_inject_timeout): launches left to inject.
static std::atomic<int> g_inject_timeout{0};

void set_injected_timeouts(int launches) { g_inject_timeout.store(launches); }

bool take_injected_timeout() {
    for (int n = g_inject_timeout.load(); n > 0; n = g_inject_timeout.load())
        if (g_inject_timeout.compare_exchange_weak(n, n - 1)) return true;
    return false;
}

}  // namespace gqa

extern "C" int gqa_attn_check(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GQA_ERR_CUDA;
    unsigned* w = gqa::status_word();
    if (!w) return GQA_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return GQA_ERR_CUDA;
    if (v != 0 && cudaMemset(w, 0, sizeof(unsigned)) != cudaSuccess) return GQA_ERR_CUDA;
    if (v & gqa::kStatusTimeout) return GQA_ERR_DEVICE_TIMEOUT;
    if (v & gqa::kStatusBadSeqlen) return GQA_ERR_DEVICE_BAD_INPUT;
    return GQA_OK;
}

extern "C" const char* gqa_attn_strerror(int code) {
    switch (code) {
        case GQA_OK: return "ok";
        case GQA_ERR_INVALID_ARG: return "invalid argument";
        case GQA_ERR_UNSUPPORTED: return "unsupported shape (d must be 64 or 128; decode: G <= 16)";
        case GQA_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
        case GQA_ERR_CUDA: return "CUDA runtime or driver error";
        case GQA_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait ran out";
        case GQA_ERR_WORKSPACE:
            return "workspace too small, misaligned, or growth needed during stream capture";
        case GQA_ERR_DEVICE_BAD_INPUT: return "a seqlen outside [0, S_max] was clamped";
        default: return "unknown error code";
    }
}

extern "C" int gqa_attn_version(void) { return 100; }
