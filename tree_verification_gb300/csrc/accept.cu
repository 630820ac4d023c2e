// Greedy lossless acceptance and KV compaction.
//
// Graft article, architecture paragraph: retrieved nodes are verified as
// ordinary proposals and the output stays lossless.  With greedy decoding a
// node is accepted iff every token on its root path is the target's argmax
// at the node before it; the deepest accepted node (lowest index on ties)
// fixes the emitted tokens (its path after the root, then the target's
// argmax there as the bonus token) and the KV rows that join the cache.
//
// Kernels:
//   argmax_part_kernel  rows of B*Kmax fp32 logits split over CTAs; each CTA
//                       streams its slice once (HBM bound) and keeps the
//                       first maximum
//   accept_kernel       one CTA per request: reduce the splits (or read the
//                       argmax the fused lm_head kernel wrote), test every
//                       node's root path, pick the deepest accepted node,
//                       write path / tokens / bonus and advance L
//   compact_kernel      one CTA per (layer, request): copy the accepted
//                       nodes' K and V rows to the end of the cache
#include <climits>

#include "common.cuh"

namespace graft {
namespace {

constexpr int kArgThreads = 256;
constexpr int kChunk = 16384;  // logits per argmax CTA (64 KB)

struct ArgPart {
    float v;
    int id;
};

struct AcceptWs {
    ArgPart* parts;   // [B*Kmax][S]
    int32_t* L_old;   // [B] cache length before this step
    int32_t* ncopy;   // [B] rows to compact (0 when the request overflowed)
};

__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia < ib);
}

__global__ void __launch_bounds__(kArgThreads)
argmax_part_kernel(const float* __restrict__ logits, int V, int S, int chunk, ArgPart* __restrict__ parts) {
    griddep_enter();
    const int s = blockIdx.x;
    const size_t row = blockIdx.y;
    const float* r = logits + row * (size_t)V;
    const int lo = s * chunk, hi = min(V, lo + chunk);
    float bv = -INFINITY;
    int bi = INT_MAX;
    const bool vec = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
    if (vec) {
        for (int i = lo + 4 * threadIdx.x; i < hi; i += 4 * kArgThreads) {
            const float4 x = __ldcs(reinterpret_cast<const float4*>(r + i));
            if (better(x.x, i, bv, bi)) { bv = x.x; bi = i; }
            if (better(x.y, i + 1, bv, bi)) { bv = x.y; bi = i + 1; }
            if (better(x.z, i + 2, bv, bi)) { bv = x.z; bi = i + 2; }
            if (better(x.w, i + 3, bv, bi)) { bv = x.w; bi = i + 3; }
        }
    } else {
        for (int i = lo + threadIdx.x; i < hi; i += kArgThreads) {
            const float x = __ldcs(r + i);
            if (better(x, i, bv, bi)) { bv = x; bi = i; }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    __shared__ float sv[kArgThreads / 32];
    __shared__ int si[kArgThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
    __syncthreads();
    if (warp == 0) {
        bv = lane < kArgThreads / 32 ? sv[lane] : -INFINITY;
        bi = lane < kArgThreads / 32 ? si[lane] : INT_MAX;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) parts[row * S + s] = ArgPart{bv, bi};
    }
}

__global__ void __launch_bounds__(GRAFT_MAX_KMAX)
accept_kernel(int Kmax, int S, int V, int64_t Lcap, const ArgPart* __restrict__ parts, const int32_t* __restrict__ tree_tok,
              const int32_t* __restrict__ tree_parent, const int32_t* __restrict__ tree_depth, int32_t* L,
              int32_t* argmax, int32_t* acc_len, int32_t* path, int32_t* out_tok, int32_t* bonus, AcceptWs w,
              int32_t* status) {
    griddep_enter();
    const int b = blockIdx.x, i = threadIdx.x;
    __shared__ int g_s[GRAFT_MAX_KMAX], tok_s[GRAFT_MAX_KMAX], par_s[GRAFT_MAX_KMAX];
    __shared__ int key_s[GRAFT_MAX_KMAX / 32];
    int key = -1;
    if (i < Kmax) {
        const size_t row = (size_t)b * Kmax + i;
        int bi;
        if (S == 0) {
            // argmax given (from the fused lm_head kernel)
            bi = argmax[row];
            if (bi < 0 || bi >= V) { flag_status(status, GRAFT_STATUS_TOKEN_RANGE); bi = 0; }
        } else {
            float bv = -INFINITY;
            bi = INT_MAX;
            for (int s = 0; s < S; ++s) {
                const ArgPart p = parts[row * S + s];
                if (better(p.v, p.id, bv, bi)) { bv = p.v; bi = p.id; }
            }
            if (bi == INT_MAX) bi = 0;  // only NaNs in the row
            argmax[row] = bi;
        }
        g_s[i] = bi;
        tok_s[i] = tree_tok[row];
        par_s[i] = tree_parent[row];
    }
    __syncthreads();
    if (i < Kmax) {
        bool ok = true;
        int steps = 0;
        for (int j = i; j > 0; ++steps) {
            const int p = par_s[j];
            if (p < 0 || p >= j || tok_s[j] != g_s[p]) { ok = false; break; }
            j = p;
        }
        if (ok) {
            if (steps != tree_depth[(size_t)b * Kmax + i]) flag_status(status, GRAFT_STATUS_TREE);
            key = (steps << 7) | (127 - i);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, off));
    if ((i & 31) == 0) key_s[i >> 5] = key;
    __syncthreads();
    if (i == 0) {
        key = max(key_s[0], key_s[1]);
        const int best = 127 - (key & 127);
        const int n = (key >> 7) + 1;
        int nodes[GRAFT_MAX_KMAX];
        int j = best;
        for (int t = n - 1; t >= 0; --t) { nodes[t] = j; j = par_s[j]; }
        int32_t* prow = path + (size_t)b * Kmax;
        int32_t* orow = out_tok + (size_t)b * Kmax;
        for (int t = 0; t < Kmax; ++t) {
            prow[t] = t < n ? nodes[t] : -1;
            orow[t] = t < n - 1 ? tok_s[nodes[t + 1]] : (t == n - 1 ? g_s[best] : -1);
        }
        acc_len[b] = n;
        bonus[b] = g_s[best];
        const int Lb = L[b];
        w.L_old[b] = Lb;
        int copy = n;
        if (Lb < 0 || Lb > Lcap) { flag_status(status, GRAFT_STATUS_LENGTH); copy = 0; }
        else if ((int64_t)Lb + n > Lcap) { flag_status(status, GRAFT_STATUS_CACHE_OVERFLOW); copy = 0; }
        w.ncopy[b] = copy;
        if (copy > 0) L[b] = Lb + copy;
    }
}

__global__ void __launch_bounds__(256)
compact_kernel(int Kmax, int64_t Lcap, int row_bytes, void* const* __restrict__ Kc_layers,
               void* const* __restrict__ Vc_layers, const void* const* __restrict__ Kt_layers,
               const void* const* __restrict__ Vt_layers, const int32_t* __restrict__ path, AcceptWs w) {
    griddep_enter();
    const int l = blockIdx.x, b = blockIdx.y;
    const int n = w.ncopy[b];
    if (n == 0) return;
    const int64_t L0 = w.L_old[b];
    const int32_t* prow = path + (size_t)b * Kmax;
    char* Kc = static_cast<char*>(Kc_layers[l]);
    char* Vc = static_cast<char*>(Vc_layers[l]);
    const char* Kt = static_cast<const char*>(Kt_layers[l]);
    const char* Vt = static_cast<const char*>(Vt_layers[l]);
    const bool vec = (row_bytes & 15) == 0 &&
                     ((reinterpret_cast<uintptr_t>(Kc) | reinterpret_cast<uintptr_t>(Vc) |
                       reinterpret_cast<uintptr_t>(Kt) | reinterpret_cast<uintptr_t>(Vt)) & 15) == 0;
    if (vec) {
        const int per = row_bytes / 16;
        for (int it = threadIdx.x; it < n * per; it += blockDim.x) {
            const int t = it / per, q = it % per;
            const size_t src = ((size_t)b * Kmax + prow[t]) * row_bytes + (size_t)q * 16;
            const size_t dst = ((size_t)b * Lcap + L0 + t) * row_bytes + (size_t)q * 16;
            *reinterpret_cast<uint4*>(Kc + dst) = *reinterpret_cast<const uint4*>(Kt + src);
            *reinterpret_cast<uint4*>(Vc + dst) = *reinterpret_cast<const uint4*>(Vt + src);
        }
    } else {
        const int per = row_bytes / 2;
        for (int it = threadIdx.x; it < n * per; it += blockDim.x) {
            const int t = it / per, q = it % per;
            const size_t src = ((size_t)b * Kmax + prow[t]) * row_bytes + (size_t)q * 2;
            const size_t dst = ((size_t)b * Lcap + L0 + t) * row_bytes + (size_t)q * 2;
            *reinterpret_cast<uint16_t*>(Kc + dst) = *reinterpret_cast<const uint16_t*>(Kt + src);
            *reinterpret_cast<uint16_t*>(Vc + dst) = *reinterpret_cast<const uint16_t*>(Vt + src);
        }
    }
}

int arg_splits(int V) { return (V + kChunk - 1) / kChunk; }

AcceptWs carve_accept(WsCarver& c, int B, int Kmax, int V) {
    AcceptWs w;
    w.parts = c.take<ArgPart>((size_t)B * Kmax * arg_splits(V));
    w.L_old = c.take<int32_t>(B);
    w.ncopy = c.take<int32_t>(B);
    return w;
}

}  // namespace
}  // namespace graft

using namespace graft;

extern "C" int graft_accept_compact_workspace_size(int B, int Kmax, int V, size_t* bytes) {
    if (bytes == nullptr || B < 0 || Kmax < 1 || V < 1) return GRAFT_ERR_INVALID_ARG;
    if (Kmax > GRAFT_MAX_KMAX) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    WsCarver c(nullptr);
    carve_accept(c, B, Kmax, V);
    *bytes = c.bytes();
    return GRAFT_OK;
}

extern "C" int graft_accept_compact(int B, int Kmax, int V, int n_layers, const float* target_logits,
                                    const int32_t* tree_tok, const int32_t* tree_parent, const int32_t* tree_depth,
                                    void* const* Kc_layers, void* const* Vc_layers, const void* const* Kt_layers,
                                    const void* const* Vt_layers, int Hkv, int head_dim, int64_t Lcap, int32_t* L,
                                    int32_t* argmax, int32_t* acc_len, int32_t* path, int32_t* out_tok,
                                    int32_t* bonus, int32_t* status, void* ws, size_t ws_bytes,
                                    graft_stream_t stream) {
    if (B < 0 || Kmax < 1 || V < 1 || n_layers < 0 || Hkv < 1 || head_dim < 1 || Lcap < 0)
        return GRAFT_ERR_INVALID_ARG;
    if (Kmax > GRAFT_MAX_KMAX) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    if (B == 0) return GRAFT_OK;
    if (tree_tok == nullptr || tree_parent == nullptr || tree_depth == nullptr ||
        L == nullptr || argmax == nullptr || acc_len == nullptr || path == nullptr || out_tok == nullptr ||
        bonus == nullptr)
        return GRAFT_ERR_INVALID_ARG;
    if (n_layers > 0 && (Kc_layers == nullptr || Vc_layers == nullptr || Kt_layers == nullptr || Vt_layers == nullptr))
        return GRAFT_ERR_INVALID_ARG;
    const long long rows = (long long)B * Kmax;
    const int S = target_logits != nullptr ? arg_splits(V) : 0;  // 0: argmax is an input
    if (rows > 65535 || S > 65535 || B > 65535 || n_layers > 65535) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    const long long row_bytes = (long long)Hkv * head_dim * 2;
    if (row_bytes > (1LL << 30)) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    WsCarver sizer(nullptr);
    carve_accept(sizer, B, Kmax, V);
    if (!ws_ok(ws, ws_bytes, sizer.bytes())) return GRAFT_ERR_WORKSPACE;
    WsCarver c(ws);
    AcceptWs w = carve_accept(c, B, Kmax, V);
    cudaStream_t st = (cudaStream_t)stream;
    if (S > 0) {
        launch_pdl(argmax_part_kernel, dim3(S, (unsigned)rows), dim3(kArgThreads), 0, st, target_logits, V, S, kChunk,
                   w.parts);
        count_launches(1);
    }
    launch_pdl(accept_kernel, dim3(B), dim3(GRAFT_MAX_KMAX), 0, st, Kmax, S, V, Lcap, w.parts, tree_tok, tree_parent,
               tree_depth, L, argmax, acc_len, path, out_tok, bonus, w, status);
    count_launches(n_layers > 0 ? 2 : 1);
    if (n_layers > 0)
        launch_pdl(compact_kernel, dim3(n_layers, B), dim3(256), 0, st, Kmax, Lcap, (int)row_bytes, Kc_layers, Vc_layers, Kt_layers,
                                                          Vt_layers, path, w);
    return launch_status();
}
