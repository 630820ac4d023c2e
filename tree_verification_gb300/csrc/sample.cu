// The target's sample at every tree node, for lossless sampling acceptance.
//
// Graft article, architecture paragraph, and Graft abstract: verification is
// lossless.  Every proposal in a Graft tree is deterministic (the drafter's
// top-k, retrieved successors); for such proposals the speculative-sampling
// rule over a node's children (try them in order, accept with the residual
// probability, renormalise on rejection) has the same law as drawing one
// sample y ~ softmax(logits / T) per node and accepting the first child whose
// token is y.  The sample is argmax_v(logits[v] / T + G_v) with Gumbel noise
// G keyed by position (philox.cuh); graft_accept_compact with these samples
// as its argmax input then applies the acceptance.
//
// Kernels: sample_part_kernel splits each row over CTAs (one Philox call per
// four tokens, HBM bound on the logits) and keeps the best perturbed score
// with the lower id on ties; sample_reduce_kernel merges a row's splits (one
// warp per row).
#include <climits>

#include "common.cuh"
#include "philox.cuh"

namespace graft {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 16384;  // tokens per split (a multiple of 4)

struct SamplePart {
    float z;
    int id;
};

__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia < ib);
}

__global__ void __launch_bounds__(kThreads)
sample_part_kernel(const float* __restrict__ logits, int Kmax, int V, int S, float inv_T, unsigned long long seed,
                   const int32_t* __restrict__ tree_pos, SamplePart* __restrict__ parts) {
    griddep_enter();
    const int s = blockIdx.x;
    const size_t row = blockIdx.y;
    const uint32_t b = (uint32_t)(row / Kmax);
    const uint32_t pos = (uint32_t)(tree_pos[row] + 1);  // the position of the token this node samples
    const float* r = logits + row * (size_t)V;
    const int lo = s * kChunk, hi = min(V, lo + kChunk);
    float bz = -INFINITY;
    int bi = INT_MAX;
    for (int q = lo / 4 + threadIdx.x; 4 * q < hi; q += kThreads) {
        const uint4 x = noise_draws(seed, b, pos, (uint32_t)q);
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int v = 4 * q + j;
            if (v < hi) {
                const float z = __ldcs(r + v) * inv_T + gumbel_of(xs[j]);
                if (better(z, v, bz, bi)) { bz = z; bi = v; }
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float oz = __shfl_xor_sync(0xffffffffu, bz, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (better(oz, oi, bz, bi)) { bz = oz; bi = oi; }
    }
    __shared__ float sz[kThreads / 32];
    __shared__ int si[kThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) { sz[warp] = bz; si[warp] = bi; }
    __syncthreads();
    if (warp == 0) {
        bz = lane < kThreads / 32 ? sz[lane] : -INFINITY;
        bi = lane < kThreads / 32 ? si[lane] : INT_MAX;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float oz = __shfl_xor_sync(0xffffffffu, bz, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (better(oz, oi, bz, bi)) { bz = oz; bi = oi; }
        }
        if (lane == 0) parts[row * S + s] = SamplePart{bz, bi};
    }
}

__global__ void __launch_bounds__(256)
sample_reduce_kernel(const SamplePart* __restrict__ parts, int rows, int S, int32_t* __restrict__ sampled) {
    griddep_enter();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= rows) return;
    float bz = -INFINITY;
    int bi = INT_MAX;
    for (int s = lane; s < S; s += 32) {
        const SamplePart p = parts[(size_t)warp * S + s];
        if (better(p.z, p.id, bz, bi)) { bz = p.z; bi = p.id; }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float oz = __shfl_xor_sync(0xffffffffu, bz, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (better(oz, oi, bz, bi)) { bz = oz; bi = oi; }
    }
    if (lane == 0) sampled[warp] = bi == INT_MAX ? 0 : bi;  // only NaNs: token 0
}

}  // namespace
}  // namespace graft

using namespace graft;

extern "C" int graft_sample_tokens_workspace_size(int B, int Kmax, int V, size_t* bytes) {
    if (bytes == nullptr || B < 0 || Kmax < 1 || V < 1) return GRAFT_ERR_INVALID_ARG;
    WsCarver c(nullptr);
    c.take<SamplePart>((size_t)B * Kmax * ((V + kChunk - 1) / kChunk));
    *bytes = c.bytes();
    return GRAFT_OK;
}

extern "C" int graft_sample_tokens(int B, int Kmax, int V, const float* target_logits, const int32_t* tree_pos,
                                   float temperature, uint64_t seed, int32_t* sampled, void* ws, size_t ws_bytes,
                                   graft_stream_t stream) {
    if (B < 0 || Kmax < 1 || V < 1 || !(temperature > 0.f)) return GRAFT_ERR_INVALID_ARG;
    if (B == 0) return GRAFT_OK;
    if (target_logits == nullptr || tree_pos == nullptr || sampled == nullptr) return GRAFT_ERR_INVALID_ARG;
    const long long rows = (long long)B * Kmax;
    const int S = (V + kChunk - 1) / kChunk;
    if (rows > 65535) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    WsCarver sizer(nullptr);
    sizer.take<SamplePart>((size_t)rows * S);
    if (!ws_ok(ws, ws_bytes, sizer.bytes())) return GRAFT_ERR_WORKSPACE;
    WsCarver c(ws);
    SamplePart* parts = c.take<SamplePart>((size_t)rows * S);
    cudaStream_t st = (cudaStream_t)stream;
    launch_pdl(sample_part_kernel, dim3(S, (unsigned)rows), dim3(kThreads), 0, st, target_logits, Kmax, V, S,
               1.0f / temperature, (unsigned long long)seed, tree_pos, parts);
    launch_pdl(sample_reduce_kernel, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, st, parts, (int)rows, S, sampled);
    count_launches(2);
    return launch_status();
}
