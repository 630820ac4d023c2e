// Online update of the adjacency table M from verified pairs.
//
// Graft article, method paragraph (fourth point) and architecture paragraph:
// M is refreshed continuously from the verified tree's logits.  Layout and
// rule (the pages leave both open): succ/cnt [V][W] int32, each row ranked by
// (count desc, token asc) with empty slots (-1, 0) last; a batch of
// (src -> dst) pairs adds 1 per pair to successors already present (atomic
// increments) and lets new successors compete for the row with their
// multiplicity as count; each touched row keeps its top W.
//
// Kernels (work proportional to the number of pairs, never to V):
//   clear_kernel   resets two open-addressing hash tables in the workspace
//   pairs_kernel   one thread per pair: registers the row, increments a
//                  present successor, or counts the new (src, dst) key and
//                  links it into its row's list
//   rerank_kernel  one warp per touched row: bitonic-sorts the W slots by
//                  the packed key, then inserts the new successors with a
//                  warp ballot, walking the row's list of them when it is
//                  short, else scanning the pair table 256 slots at a time
//                  (independent loads) and inserting only the candidates
//                  that beat the row's current last entry, so a token
//                  repeated across thousands of tree nodes does not turn
//                  into thousands of dependent loads; the result depends
//                  only on the multiset
#include <mutex>

#include "common.cuh"

namespace graft {
namespace {

constexpr unsigned long long kEmptyPair = ~0ull;
constexpr int kListWalk = 8;  // rows with more new successors scan the pair table instead of their list

struct UpdWs {
    unsigned long long* pair_key;  // [cap] (src << 32) | dst, kEmptyPair = free
    int32_t* pair_mult;            // [cap]
    int32_t* pair_next;            // [cap] next new pair of the same row, -1 = end
    int32_t* row_key;              // [cap] src token, -1 = free
    int32_t* row_head;             // [cap] first new pair of the row, -1 = none
    int32_t* row_ncand;            // [cap] new successors of the row
    int32_t* touched;              // [n] row-table slots in arrival order
    int32_t* n_touched;            // [1]
    int cap;                       // power of two >= 2n
};

__device__ __forceinline__ uint32_t hash32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352dU;
    x ^= x >> 15;
    x *= 0x846ca68bU;
    x ^= x >> 16;
    return x;
}
__device__ __forceinline__ uint32_t hash64(unsigned long long x) {
    x ^= x >> 33;
    x *= 0xff51afd7ed558ccdULL;
    x ^= x >> 33;
    x *= 0xc4ceb9fe1a85ec53ULL;
    x ^= x >> 33;
    return (uint32_t)x;
}

__global__ void clear_kernel(UpdWs w) {
    griddep_enter();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < w.cap; i += gridDim.x * blockDim.x) {
        w.pair_key[i] = kEmptyPair;
        w.pair_mult[i] = 0;
        w.pair_next[i] = -1;
        w.row_key[i] = -1;
        w.row_head[i] = -1;
        w.row_ncand[i] = 0;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) *w.n_touched = 0;
}

__global__ void pairs_kernel(int32_t* __restrict__ succ, int32_t* __restrict__ cnt, int V, int W,
                             const int32_t* __restrict__ src, const int32_t* __restrict__ dst, int64_t n, UpdWs w,
                             int32_t* status) {
    griddep_enter();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int s = src[i], t = dst[i];
    if (s == -1) return;  // an empty slot or an empty tree node: no pair
    if (s < 0 || s >= V || t < 0 || t >= V) {
        flag_status(status, GRAFT_STATUS_TOKEN_RANGE);
        return;
    }
    const uint32_t mask = (uint32_t)w.cap - 1;
    // register the row (probes end: the table has at least 2n free slots)
    uint32_t h = hash32((uint32_t)s) & mask;
    for (int probe = 0; probe < w.cap; ++probe) {
        const int old = atomicCAS(&w.row_key[h], -1, s);
        if (old == -1) {
            w.touched[atomicAdd(w.n_touched, 1)] = (int)h;
            break;
        }
        if (old == s) break;
        h = (h + 1) & mask;
    }
    const int row_slot = (int)h;
    // successor already present: one atomic increment
    const int32_t* rs = succ + (size_t)s * W;
    for (int j = 0; j < W; ++j) {
        if (rs[j] == t) {
            atomicAdd(cnt + (size_t)s * W + j, 1);
            return;
        }
    }
    // new successor: count the (s, t) key; its first arrival links it into the row's list
    const unsigned long long key = ((unsigned long long)(uint32_t)s << 32) | (uint32_t)t;
    uint32_t q = hash64(key) & mask;
    for (int probe = 0; probe < w.cap; ++probe) {
        const unsigned long long old = atomicCAS(&w.pair_key[q], kEmptyPair, key);
        if (old == kEmptyPair) {
            w.pair_next[q] = atomicExch(&w.row_head[row_slot], (int)q);
            atomicAdd(&w.row_ncand[row_slot], 1);
            atomicAdd(&w.pair_mult[q], 1);
            return;
        }
        if (old == key) {
            atomicAdd(&w.pair_mult[q], 1);
            return;
        }
        q = (q + 1) & mask;
    }
}

// Packs a slot so that a smaller key ranks first: count desc, then token asc.
// Empty slots (cnt 0, token -1) sort after every real entry; lanes past W
// carry count -1 and sort after the empties.
__device__ __forceinline__ unsigned long long pack_slot(int c, int tok) {
    return ((unsigned long long)(uint32_t)(0x7fffffff - c) << 32) | (uint32_t)tok;
}

__global__ void rerank_kernel(int32_t* __restrict__ succ, int32_t* __restrict__ cnt, int W, UpdWs w) {
    griddep_enter();
    const int warps = blockDim.x >> 5;
    const int wid = blockIdx.x * warps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (wid >= *w.n_touched) return;
    const int slot = w.touched[wid];
    const int s = w.row_key[slot];
    int32_t* rs = succ + (size_t)s * W;
    int32_t* rc = cnt + (size_t)s * W;
    unsigned long long key = lane < W ? pack_slot(rc[lane], rs[lane]) : pack_slot(-1, -1);
    // bitonic sort, ascending key
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, j);
            const bool up = (lane & k) == 0;
            const bool lower = (lane & j) == 0;
            const unsigned long long lo = key < other ? key : other;
            const unsigned long long hi = key < other ? other : key;
            key = (lower == up) ? lo : hi;
        }
    }
    // insert the row's new successors (order of insertion does not matter): a candidate enters at the
    // number of entries ranked ahead of it, if that is below W, shifting the rest down one
    auto insert = [&](unsigned long long ck) {
        const unsigned ahead = __ballot_sync(0xffffffffu, key < ck);
        const int pos = __popc(ahead);  // entries that stay in front (a prefix, the list is sorted)
        if (pos < W) {
            const unsigned long long prev = __shfl_up_sync(0xffffffffu, key, 1);
            if (lane > pos) key = prev;
            else if (lane == pos) key = ck;
        }
    };
    if (w.row_ncand[slot] <= kListWalk) {
        for (int p = w.row_head[slot]; p >= 0; p = w.pair_next[p])
            insert(pack_slot(w.pair_mult[p], (int)(uint32_t)(w.pair_key[p] & 0xffffffffull)));
    } else {
        // many new successors: every pair-table slot is read once, eight independent loads per lane per
        // pass, and a candidate is inserted only if it ranks ahead of the row's current W-th entry
        const unsigned long long row_src = (unsigned long long)(uint32_t)s;
        for (int base = 0; base < w.cap; base += 8 * 32) {
            unsigned long long kk[8];
            int mm[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int q = base + u * 32 + lane;
                kk[u] = q < w.cap ? w.pair_key[q] : kEmptyPair;
                mm[u] = q < w.cap ? w.pair_mult[q] : 0;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const bool mine = kk[u] != kEmptyPair && (kk[u] >> 32) == row_src;
                const unsigned long long ck = mine ? pack_slot(mm[u], (int)(uint32_t)(kk[u] & 0xffffffffull)) : ~0ull;
                const unsigned long long last = __shfl_sync(0xffffffffu, key, W - 1);
                unsigned want = __ballot_sync(0xffffffffu, ck < last);
                while (want) {
                    const int from = __ffs(want) - 1;
                    want &= want - 1;
                    insert(__shfl_sync(0xffffffffu, ck, from));
                }
            }
        }
    }
    if (lane < W) {
        const int c = 0x7fffffff - (int)(key >> 32);
        const int tok = (int)(uint32_t)(key & 0xffffffffull);
        rs[lane] = tok;
        rc[lane] = c;
    }
}

// The bigrams of the tokens a verify step emitted, one slot per tree node:
// slot t < acc_len[b] holds (previous token -> out_tok[b][t]), where the token
// before out_tok[b][0] is the tree's root (the last token emitted before the
// step); the remaining slots hold the (-1, -1) no-pair marker.
__global__ void emitted_pairs_kernel(int B, int Kmax, const int32_t* __restrict__ tree_tok,
                                     const int32_t* __restrict__ out_tok, const int32_t* __restrict__ acc_len,
                                     int32_t* __restrict__ src, int32_t* __restrict__ dst) {
    griddep_enter();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= B * Kmax) return;
    const int b = i / Kmax, t = i % Kmax;
    const int n = acc_len[b];
    if (t < n && n <= Kmax) {
        src[i] = t == 0 ? tree_tok[(size_t)b * Kmax] : out_tok[i - 1];
        dst[i] = out_tok[i];
    } else {
        src[i] = -1;
        dst[i] = -1;
    }
}

int table_cap(int64_t n) {
    int64_t cap = 64;
    while (cap < 2 * n) cap <<= 1;
    return (int)cap;
}

UpdWs carve_update(WsCarver& c, int64_t n) {
    UpdWs w;
    w.cap = table_cap(n);
    w.pair_key = c.take<unsigned long long>(w.cap);
    w.pair_mult = c.take<int32_t>(w.cap);
    w.pair_next = c.take<int32_t>(w.cap);
    w.row_key = c.take<int32_t>(w.cap);
    w.row_head = c.take<int32_t>(w.cap);
    w.row_ncand = c.take<int32_t>(w.cap);
    w.touched = c.take<int32_t>(n > 0 ? n : 1);
    w.n_touched = c.take<int32_t>(1);
    return w;
}

}  // namespace
}  // namespace graft

using namespace graft;

extern "C" int graft_update_M_workspace_size(int64_t n, size_t* bytes) {
    if (bytes == nullptr || n < 0) return GRAFT_ERR_INVALID_ARG;
    if (n > (1LL << 28)) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    WsCarver c(nullptr);
    carve_update(c, n);
    *bytes = c.bytes();
    return GRAFT_OK;
}

extern "C" int graft_update_M(int32_t* M_succ, int32_t* M_cnt, int V, int W, const int32_t* src, const int32_t* dst,
                              int64_t n, int32_t* status, void* ws, size_t ws_bytes, graft_stream_t stream) {
    if (V < 1 || W < 1 || n < 0) return GRAFT_ERR_INVALID_ARG;
    if (W > GRAFT_MAX_W || n > (1LL << 28)) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    if (n == 0) return GRAFT_OK;
    if (M_succ == nullptr || M_cnt == nullptr || src == nullptr || dst == nullptr) return GRAFT_ERR_INVALID_ARG;
    WsCarver sizer(nullptr);
    carve_update(sizer, n);
    if (!ws_ok(ws, ws_bytes, sizer.bytes())) return GRAFT_ERR_WORKSPACE;
    WsCarver c(ws);
    UpdWs w = carve_update(c, n);
    cudaStream_t st = (cudaStream_t)stream;
    const int cb = (int)((w.cap + 255) / 256);
    launch_pdl(clear_kernel, dim3(cb < 1024 ? cb : 1024), dim3(256), 0, st, w);
    launch_pdl(pairs_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, M_succ, M_cnt, V, W, src, dst, n, w, status);
    launch_pdl(rerank_kernel, dim3((unsigned)((n + 7) / 8)), dim3(256), 0, st, M_succ, M_cnt, W, w);
    count_launches(3);
    return launch_status();
}

// ----------------------------------------------------------------------------
// graft_update_M_noalloc: the same update, with its scratch in a fixed device
// array instead of a caller workspace.
//
// Some callers cannot hand the library a workspace: a plug-in that only sees
// the tensors its host framework gives it and has no device allocator of its
// own, or a latency-critical serving loop that must not call cudaMalloc
// (which synchronises the whole device).  For them the hash tables live in
// g_update_scratch below, sized for GRAFT_NOALLOC_MAX_PAIRS pairs; every GPU
// that loads the library keeps this 1 MiB until the process exits.
// ----------------------------------------------------------------------------
namespace graft {
namespace {

constexpr size_t kNoAllocScratchBytes = 1u << 20;
static __device__ __align__(256) unsigned char g_update_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[64] = {nullptr};

// Device address of g_update_scratch on the current device, looked up once
// per device.  In host code the array's name is only a host-side handle, so
// kernels must be given the address cudaGetSymbolAddress returns.
int noalloc_scratch(void** out) {
    int dev = 0;
    if (!cuda_ok(cudaGetDevice(&dev))) return GRAFT_ERR_CUDA;
    if (dev < 0 || dev >= 64) return GRAFT_ERR_UNSUPPORTED_SHAPE;  // device ordinals 0..63 (graft.h)
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (!cuda_ok(cudaGetSymbolAddress(&p, g_update_scratch))) return GRAFT_ERR_CUDA;
        if (p == nullptr) return GRAFT_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return GRAFT_OK;
}

}  // namespace
}  // namespace graft

extern "C" int graft_update_M_noalloc(int32_t* M_succ, int32_t* M_cnt, int V, int W, const int32_t* src,
                                      const int32_t* dst, int64_t n, int32_t* status, graft_stream_t stream) {
    if (V < 1 || W < 1 || n < 0) return GRAFT_ERR_INVALID_ARG;
    if (W > GRAFT_MAX_W || n > GRAFT_NOALLOC_MAX_PAIRS) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    if (n == 0) return GRAFT_OK;
    if (M_succ == nullptr || M_cnt == nullptr || src == nullptr || dst == nullptr) return GRAFT_ERR_INVALID_ARG;
    WsCarver sizer(nullptr);
    carve_update(sizer, n);
    if (sizer.bytes() > kNoAllocScratchBytes) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    void* scratch = nullptr;
    const int rc = noalloc_scratch(&scratch);
    if (rc != GRAFT_OK) return rc;
    WsCarver c(scratch);
    UpdWs w = carve_update(c, n);
    cudaStream_t st = (cudaStream_t)stream;
    // clear_kernel resets every table the other two kernels read, so whatever
    // the previous call left in the shared array does not leak into this one
    const int cb = (int)((w.cap + 255) / 256);
    launch_pdl(clear_kernel, dim3(cb < 1024 ? cb : 1024), dim3(256), 0, st, w);
    launch_pdl(pairs_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, M_succ, M_cnt, V, W, src, dst, n, w, status);
    launch_pdl(rerank_kernel, dim3((unsigned)((n + 7) / 8)), dim3(256), 0, st, M_succ, M_cnt, W, w);
    count_launches(3);
    return launch_status();
}

// ----------------------------------------------------------------------------
// graft_update_M_emitted: prompt-evidence refresh from a step's emitted tokens
// ----------------------------------------------------------------------------
extern "C" int graft_update_M_emitted_workspace_size(int B, int Kmax, size_t* bytes) {
    if (bytes == nullptr || B < 0 || Kmax < 1) return GRAFT_ERR_INVALID_ARG;
    const int64_t n = (int64_t)B * Kmax;
    if (n > (1LL << 28)) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    WsCarver c(nullptr);
    c.take<int32_t>(n);
    c.take<int32_t>(n);
    carve_update(c, n);
    *bytes = c.bytes();
    return GRAFT_OK;
}

extern "C" int graft_update_M_emitted(int32_t* M_succ, int32_t* M_cnt, int V, int W, int B, int Kmax,
                                      const int32_t* tree_tok, const int32_t* out_tok, const int32_t* acc_len,
                                      int32_t* status, void* ws, size_t ws_bytes, graft_stream_t stream) {
    if (V < 1 || W < 1 || B < 0 || Kmax < 1) return GRAFT_ERR_INVALID_ARG;
    if (W > GRAFT_MAX_W || Kmax > GRAFT_MAX_KMAX) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    if (B == 0) return GRAFT_OK;
    if (M_succ == nullptr || M_cnt == nullptr || tree_tok == nullptr || out_tok == nullptr || acc_len == nullptr)
        return GRAFT_ERR_INVALID_ARG;
    const int64_t n = (int64_t)B * Kmax;
    if (n > (1LL << 28)) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    size_t need = 0;
    graft_update_M_emitted_workspace_size(B, Kmax, &need);
    if (!ws_ok(ws, ws_bytes, need)) return GRAFT_ERR_WORKSPACE;
    WsCarver c(ws);
    int32_t* src = c.take<int32_t>(n);
    int32_t* dst = c.take<int32_t>(n);
    UpdWs w = carve_update(c, n);
    cudaStream_t st = (cudaStream_t)stream;
    const int cb = (int)((w.cap + 255) / 256);
    launch_pdl(emitted_pairs_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, B, Kmax, tree_tok, out_tok,
               acc_len, src, dst);
    launch_pdl(clear_kernel, dim3(cb < 1024 ? cb : 1024), dim3(256), 0, st, w);
    launch_pdl(pairs_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, M_succ, M_cnt, V, W, src, dst, n,
               w, status);
    launch_pdl(rerank_kernel, dim3((unsigned)((n + 7) / 8)), dim3(256), 0, st, M_succ, M_cnt, W, w);
    count_launches(4);
    return launch_status();
}
