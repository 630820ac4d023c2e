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
// Kernels: sample_part_kernel splits each row over CTAs, reads its split's
// logits once, draws noise (one Philox call per four tokens) only for groups
// that can still hold the split's pick, and keeps the best perturbed score
// with the lower id on ties; sample_reduce_kernel merges a row's splits (one
// warp per row).
#include <climits>

#include "common.cuh"
#include "philox.cuh"

namespace graft {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 8192;  // tokens per split (a multiple of 4 kThreads)

struct SamplePart {
    float z;
    int id;
};

__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia < ib);
}

constexpr int kGroups = kChunk / (4 * kThreads);  // four-token groups per thread and split
static_assert(kChunk % (4 * kThreads) == 0, "a split is whole four-token groups of every thread");

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
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // The split's scaled logits, read once (group g of this thread: tokens 4 q .. 4 q + 3 with
    // q = lo / 4 + threadIdx.x + g kThreads; -inf past the row), and their maximum.
    const bool vec = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
    float4 xs[kGroups];
    if (vec && hi - lo == kChunk) {
        // a whole aligned split: every load issued before any is used
#pragma unroll
        for (int g = 0; g < kGroups; ++g)
            xs[g] = __ldcs(reinterpret_cast<const float4*>(r + 4 * (lo / 4 + (int)threadIdx.x + g * kThreads)));
    } else {
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
            const int v = 4 * (lo / 4 + (int)threadIdx.x + g * kThreads);
            xs[g].x = v < hi ? __ldcs(r + v) : -INFINITY;
            xs[g].y = v + 1 < hi ? __ldcs(r + v + 1) : -INFINITY;
            xs[g].z = v + 2 < hi ? __ldcs(r + v + 2) : -INFINITY;
            xs[g].w = v + 3 < hi ? __ldcs(r + v + 3) : -INFINITY;
        }
    }
    float m = -INFINITY;
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
        const float4 x = make_float4(xs[g].x * inv_T, xs[g].y * inv_T, xs[g].z * inv_T, xs[g].w * inv_T);
        xs[g] = x;
        m = fmaxf(m, fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)));
    }
    __shared__ float sm[kThreads / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) sm[warp] = m;
    __syncthreads();
    m = sm[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, sm[w]);
    // Every token's score is its scaled logit plus a draw of at least g_bot, so the split's best score
    // is at least m + g_bot; a group whose scaled logits plus the largest draw (g_top) stay below that
    // cannot hold the split's pick and draws no noise.  The margins allow for the rounding of the
    // logarithms and of the sums; without a finite bound nothing is skipped.
    const float g_top = gumbel_of(0xffffffffu) + 1e-3f, g_bot = gumbel_of(0u) - 1e-3f;
    const float floor_score = m + g_bot;
    const float lim = fabsf(floor_score) < INFINITY
                          ? floor_score - g_top - fabsf(floor_score) * 9.5367431640625e-7f
                          : -INFINITY;
    float bz = -INFINITY;
    int bi = INT_MAX;
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
        const int q = lo / 4 + threadIdx.x + g * kThreads;
        const float4 x = xs[g];
        if (4 * q < hi && fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)) >= lim) {
            const uint4 d = noise_draws(seed, b, pos, (uint32_t)q);
            const float z[4] = {x.x + gumbel_of(d.x), x.y + gumbel_of(d.y), x.z + gumbel_of(d.z),
                                x.w + gumbel_of(d.w)};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int v = 4 * q + j;
                if (v < hi && better(z[j], v, bz, bi)) { bz = z[j]; bi = v; }
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
