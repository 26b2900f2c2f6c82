// smla_decode_static_scratch: the decode entry point for callers that cannot
// allocate device memory.
//
// Some callers have no way to call cudaMalloc.  Examples: a plugin or
// custom-op interface that hands the kernel only its inputs, its outputs and a
// stream; code that runs while a CUDA graph is being captured, where cudaMalloc
// is not a stream operation and cannot be recorded; and processes whose device
// memory is entirely owned by another allocator.  For them the scratch that
// smla_decode takes as a caller-owned workspace lives here instead, in a
// file-scope __device__ array of SMLA_STATIC_SCRATCH_BYTES that every GPU
// which loads the library holds until the process exits.
//
// Host code must not pass the array's name to a kernel: on the host it is
// only a stand-in symbol, not a device address.  The device address is
// looked up once per device with cudaGetSymbolAddress (with that device
// current) on the first call made on that device, and cached.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "smla.h"
#include "smla_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_smla_scratch[SMLA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_smla_scratch on the current device (looked up once),
// after the device check: on a device that is not sm_103 the call returns
// SMLA_ERR_UNSUPPORTED_DEVICE, as smla_decode does.
smla_status scratch_on_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SMLA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SMLA_ERR_UNSUPPORTED_DEVICE;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return SMLA_ERR_CUDA;
    if (major != 10 || minor != 3) return SMLA_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_smla_scratch);
        if (e != cudaSuccess || p == nullptr) return SMLA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SMLA_OK;
}

}  // namespace

extern "C" smla_status smla_decode_static_scratch(const smla_decode_args* args, smla_stream_t stream) {
    // Every host check runs before the array is touched: a rejected call
    // leaves the array (and the GPU) alone.
    if (args == nullptr) return SMLA_ERR_NULL_POINTER;
    const size_t need = smla_workspace_bytes(args->num_rows, args->num_heads, args->num_splits);
    if (need == 0) return SMLA_ERR_BAD_SHAPE;
    if (need > (size_t)SMLA_STATIC_SCRATCH_BYTES) return SMLA_ERR_WORKSPACE_TOO_SMALL;
    smla_status st = smla::check_decode_args(args);
    if (st != SMLA_OK) return st;
    void* scratch = nullptr;
    st = scratch_on_current_device(&scratch);  // checks the device first
    if (st != SMLA_OK) return st;
    st = smla::check_decode_call(args, scratch, (size_t)SMLA_STATIC_SCRATCH_BYTES);
    if (st != SMLA_OK) return st;
    // The error word must start at zero.  The array keeps whatever the
    // previous call left, so clear the head of the layout on the stream.
    const smla::WorkspaceLayout L = smla::workspace_layout(args->num_rows, args->num_heads, args->num_splits);
    if (cudaMemsetAsync(scratch, 0, L.off_ml, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SMLA_ERR_CUDA;
    return smla::launch_decode(args, scratch, static_cast<cudaStream_t>(stream));
}
