// Shared device helpers for the graft kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

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

inline int launch_status() {
    return cudaGetLastError() == cudaSuccess ? GRAFT_OK : GRAFT_ERR_CUDA;
}

// Counts kernel launches enqueued by the library (graft_launch_count).
void count_launches(int n);

// Number of SMs of the current device (cached per device ordinal).
int device_sm_count();

}  // namespace graft
