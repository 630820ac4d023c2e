// Shared device helpers for the graft kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "graft.h"

namespace graft {

constexpr int kWarp = 32;
constexpr size_t kWsAlign = 256;

__device__ __forceinline__ void flag_status(int32_t* status, int bits) {
    if (status != nullptr) atomicOr(status, bits);
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Carves typed sub-buffers out of a caller workspace.  The same sequence of
// take() calls is run once with base == nullptr to size the workspace.
struct WsCarver {
    char* base;
    size_t off = 0;
    explicit WsCarver(void* b) : base(static_cast<char*>(b)) {}
    template <class T>
    T* take(size_t n) {
        off = align_up(off, kWsAlign);
        T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
        off += n * sizeof(T);
        return p;
    }
    size_t bytes() const { return align_up(off, kWsAlign); }
};

inline bool ws_ok(const void* ws, size_t have, size_t need) {
    if (need == 0) return true;
    if (ws == nullptr || have < need) return false;
    return (reinterpret_cast<uintptr_t>(ws) % kWsAlign) == 0;
}

// Records a CUDA runtime error for graft_last_cuda_error (per host thread).
void note_cuda_error(cudaError_t e);

inline bool cuda_ok(cudaError_t e) {
    if (e == cudaSuccess) return true;
    note_cuda_error(e);
    return false;
}

inline int launch_status() {
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return GRAFT_OK;
    note_cuda_error(e);
    return GRAFT_ERR_CUDA;
}

// Counts kernel launches enqueued by the library (graft_launch_count).
void count_launches(int n);

// Programmatic dependent launch.  Every library kernel is launched with
// programmatic stream serialisation: it may become resident while its
// predecessor in the stream is still running, does only work that touches
// no global memory (barrier set-up, tensor-memory allocation) before
// griddep_wait(), which returns once the predecessor has completed and its
// writes are visible, and then lets its own successor launch early.  Waits
// chain, so a kernel also sees everything earlier kernels wrote.  After an
// ordinary launch both instructions are no-ops.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Both at once, for kernels with no prologue worth overlapping.
__device__ __forceinline__ void griddep_enter() {
    griddep_wait();
    griddep_launch_dependents();
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Number of SMs of the current device (cached per device ordinal).
int device_sm_count();

}  // namespace graft
