// Stages 1-3 of the verify step: draft tree with dynamic-depth pruning,
// retrieval fill from M, and the hybrid merge.
//
// Graft article, step summary and method paragraph (first three points);
// architecture paragraph (checkpoints d0/d1/d5, Kmax = K_draft_s + K_ret_s,
// |T_s| = Kmax, per-stage template prefixes); Graft abstract
// ("prune-then-graft" fills the positions pruning opened).
//
// Kernel plan (all on the caller's stream, no host round trip):
//   retrieve_kernel       one CTA per request, one thread per envelope node,
//                         level by level through M (independent of drafting)
//   for each checkpoint group g (drafter calls between two checkpoints):
//     draft_rows_kernel   streams the group's logit rows once: per row split,
//                         online log-sum-exp and a register top-k (HBM bound)
//     draft_select_kernel one CTA per request: combines the splits, scores
//                         the children, picks the next frontier, computes
//                         c_d and applies the gate at the checkpoint
//   draft_merge_kernel    one CTA per request: reranks the pool, orders the
//                         kept draft, appends the stage's envelope prefix and
//                         writes parents, depths, positions and ancestor masks
// Requests pruned at an earlier checkpoint skip later groups, so rows past
// the pruning point are never read.
#include <climits>
#include <cmath>

#include "common.cuh"

namespace graft {
namespace {

constexpr int kRowThreads = 256;
constexpr int kSelThreads = 256;
constexpr int kMaxSplits = 32;

struct RowPart {
    float m;    // running max of the split
    float s;    // sum of exp(x - m) over the split
    float v[GRAFT_MAX_TOPK];
    int id[GRAFT_MAX_TOPK];
};

__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia < ib);
}

template <int KT>
struct TopK {
    float v[KT];
    int id[KT];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int j = 0; j < KT; ++j) { v[j] = -INFINITY; id[j] = INT_MAX; }
    }
    __device__ __forceinline__ void offer(float x, int i) {
        if (!better(x, i, v[KT - 1], id[KT - 1])) return;
#pragma unroll
        for (int j = KT - 1; j >= 0; --j) {
            const bool here = better(x, i, v[j], id[j]);
            const bool above = (j > 0) && better(x, i, v[j - 1], id[j - 1]);
            if (here) {
                if (above) { v[j] = v[j - 1]; id[j] = id[j - 1]; }
                else { v[j] = x; id[j] = i; }
            }
        }
    }
    __device__ __forceinline__ void pop() {
#pragma unroll
        for (int j = 0; j < KT - 1; ++j) { v[j] = v[j + 1]; id[j] = id[j + 1]; }
        v[KT - 1] = -INFINITY;
        id[KT - 1] = INT_MAX;
    }
};

// Merge (m, s) log-sum-exp partials.
__device__ __forceinline__ void lse_merge(float& m, float& s, float om, float os) {
    if (om > m) {
        s = s * __expf(m - om) + os;
        m = om;
    } else if (om > -INFINITY) {
        s += os * __expf(om - m);
    }
}

// Warp-wide k-round tournament: lane 0 ends with the warp's best KT entries in out_v/out_id.
template <int KT>
__device__ __forceinline__ void warp_topk(TopK<KT>& tk, float* out_v, int* out_id) {
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int r = 0; r < KT; ++r) {
        float bv = tk.v[0];
        int bi = tk.id[0];
        int bl = lane;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            const int ol = __shfl_xor_sync(0xffffffffu, bl, off);
            if (better(ov, oi, bv, bi) || (ov == bv && oi == bi && ol < bl)) { bv = ov; bi = oi; bl = ol; }
        }
        if (lane == 0) { out_v[r] = bv; out_id[r] = bi; }
        if (lane == bl) tk.pop();
    }
}

template <int KT>
__global__ void __launch_bounds__(kRowThreads)
draft_rows_kernel(const float* __restrict__ logits, int D, int k, int V, int d_lo, int S,
                  int chunk, const int32_t* __restrict__ state, RowPart* __restrict__ parts, int block) {
    griddep_enter();
    const int s = blockIdx.x;
    const int r = blockIdx.y;
    const int b = blockIdx.z;
    const int d = d_lo + r / k;
    const int f = r % k;
    if (d >= D || (d == 0 && f != 0)) return;
    if (state != nullptr && state[b] != -1) return;  // pruned at an earlier checkpoint

    // the split's result goes to slot (b, d, f); block drafts read one row per depth, shared by
    // every frontier node of that depth
    const size_t row_id = ((size_t)b * D + d) * k + f;
    const size_t in_row = block ? (size_t)b * D + d : row_id;
    const float* row = logits + in_row * (size_t)V;
    const int lo = s * chunk;
    const int hi = min(V, lo + chunk);

    float m = -INFINITY, sum = 0.f;
    TopK<KT> tk;
    tk.init();
    auto take = [&](float x, int i) {
        if (x > m) {
            sum = sum * __expf(m - x) + 1.f;
            m = x;
        } else if (x > -INFINITY) {
            sum += __expf(x - m);
        }
        tk.offer(x, i);
    };
    const bool vec = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
    if (vec) {
        for (int i = lo + 4 * threadIdx.x; i < hi; i += 4 * kRowThreads) {
            const float4 x = __ldcs(reinterpret_cast<const float4*>(row + i));
            take(x.x, i);
            take(x.y, i + 1);
            take(x.z, i + 2);
            take(x.w, i + 3);
        }
    } else {
        for (int i = lo + threadIdx.x; i < hi; i += kRowThreads) take(__ldcs(row + i), i);
    }

    __shared__ float sm_m[kRowThreads / 32], sm_s[kRowThreads / 32];
    __shared__ float sm_v[kRowThreads / 32][KT];
    __shared__ int sm_id[kRowThreads / 32][KT];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, off);
        const float os = __shfl_xor_sync(0xffffffffu, sum, off);
        lse_merge(m, sum, om, os);
    }
    warp_topk<KT>(tk, sm_v[warp], sm_id[warp]);
    if (lane == 0) { sm_m[warp] = m; sm_s[warp] = sum; }
    __syncthreads();
    if (warp != 0) return;
    constexpr int NW = kRowThreads / 32;
    m = lane < NW ? sm_m[lane] : -INFINITY;
    sum = lane < NW ? sm_s[lane] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, off);
        const float os = __shfl_xor_sync(0xffffffffu, sum, off);
        lse_merge(m, sum, om, os);
    }
    TopK<KT> wk;
    wk.init();
    if (lane < NW) {
#pragma unroll
        for (int j = 0; j < KT; ++j) { wk.v[j] = sm_v[lane][j]; wk.id[j] = sm_id[lane][j]; }
    }
    __shared__ float fin_v[KT];
    __shared__ int fin_id[KT];
    warp_topk<KT>(wk, fin_v, fin_id);
    __syncwarp();
    RowPart* out = parts + row_id * S + s;
    if (lane == 0) { out->m = m; out->s = sum; }
    if (lane < k) { out->v[lane] = fin_v[lane]; out->id[lane] = fin_id[lane]; }
}

struct SelectParams {
    int D, k, S, n_cp;
    int checkpoint[GRAFT_MAX_CHECKPOINTS];
    float tau[GRAFT_MAX_CHECKPOINTS];
};

struct BuildWs {
    RowPart* parts;       // [B][D][k][S]
    float* pool_score;    // [B][D][k*k]
    int32_t* pool_tok;    // [B][D][k*k]
    int32_t* pool_par;    // [B][D][k*k] parent's index among its depth's candidates (-1 = root)
    int32_t* front_idx;   // [B][MAX_TOPK]
    float* front_score;   // [B][MAX_TOPK]
    int32_t* state;       // [B] -1 = still drafting, else the stage
    float* conf;          // [B][D] c_d
    int32_t* ret;         // [B][MAX_KMAX] envelope tokens (-1 = pad)
};

__global__ void __launch_bounds__(kSelThreads)
draft_select_kernel(SelectParams p, int d_lo, int d_hi, BuildWs w) {
    griddep_enter();
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NW = kSelThreads / 32;
    const int k = p.k, D = p.D, S = p.S;
    const int KK = k * k;

    __shared__ float lse_s[GRAFT_MAX_TOPK];
    __shared__ float top_v[GRAFT_MAX_TOPK][GRAFT_MAX_TOPK];
    __shared__ int top_id[GRAFT_MAX_TOPK][GRAFT_MAX_TOPK];
    __shared__ float cand_score[GRAFT_MAX_TOPK * GRAFT_MAX_TOPK];
    __shared__ int front_idx[GRAFT_MAX_TOPK];
    __shared__ float front_score[GRAFT_MAX_TOPK];
    __shared__ int new_idx[GRAFT_MAX_TOPK];
    __shared__ float new_score[GRAFT_MAX_TOPK];
    __shared__ int st;

    if (d_lo > 0) {
        if (w.state[b] != -1) return;
        if (tid < k) {
            front_idx[tid] = w.front_idx[b * GRAFT_MAX_TOPK + tid];
            front_score[tid] = w.front_score[b * GRAFT_MAX_TOPK + tid];
        }
    }
    if (tid == 0) st = -1;
    __syncthreads();

    for (int d = d_lo; d <= d_hi; ++d) {
        const int np = (d == 0) ? 1 : k;
        // combine the splits of every parent row of this call
        for (int f = warp; f < np; f += NW) {
            const RowPart* rp = w.parts + (((size_t)b * D + d) * k + f) * S;
            float m = -INFINITY, sum = 0.f;
            for (int s = lane; s < S; s += 32) lse_merge(m, sum, rp[s].m, rp[s].s);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float om = __shfl_xor_sync(0xffffffffu, m, off);
                const float os = __shfl_xor_sync(0xffffffffu, sum, off);
                lse_merge(m, sum, om, os);
            }
            // S <= 32 sorted lists, one per lane: k-round tournament
            int ptr = 0;
            for (int r = 0; r < k; ++r) {
                float bv = -INFINITY;
                int bi = INT_MAX;
                if (lane < S && ptr < k) { bv = rp[lane].v[ptr]; bi = rp[lane].id[ptr]; }
                int bl = lane;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                    const int ol = __shfl_xor_sync(0xffffffffu, bl, off);
                    if (better(ov, oi, bv, bi) || (ov == bv && oi == bi && ol < bl)) { bv = ov; bi = oi; bl = ol; }
                }
                if (lane == 0) { top_v[f][r] = bv; top_id[f][r] = bi; }
                if (lane == bl) ++ptr;
            }
            if (lane == 0) lse_s[f] = m + logf(sum);
        }
        __syncthreads();
        // score every child: parent score + (logit - lse), single float32 operations
        const int nc = np * k;
        for (int c = tid; c < nc; c += kSelThreads) {
            const int f = c / k, r = c % k;
            const float ps = (d == 0) ? 0.f : front_score[f];
            float sc = __fadd_rn(ps, __fsub_rn(top_v[f][r], lse_s[f]));
            // a non-finite row (NaN, or fewer than k finite logits) yields the lowest score and a
            // pad token, so every ranking below stays a strict total order
            int tok = top_id[f][r];
            if (!(sc == sc) || tok == INT_MAX) sc = -INFINITY;
            if (tok == INT_MAX) tok = 0;
            cand_score[c] = sc;
            const size_t o = ((size_t)b * D + d) * KK + c;
            w.pool_score[o] = sc;
            w.pool_tok[o] = tok;
            w.pool_par[o] = (d == 0) ? -1 : front_idx[f];
        }
        __syncthreads();
        // next frontier: the k best by (score desc, index asc)
        for (int c = tid; c < nc; c += kSelThreads) {
            const float sc = cand_score[c];
            int rank = 0;
            for (int c2 = 0; c2 < nc; ++c2) {
                const float o = cand_score[c2];
                rank += (o > sc) || (o == sc && c2 < c);
            }
            if (rank < k) { new_idx[rank] = c; new_score[rank] = sc; }
        }
        __syncthreads();
        if (tid < k) { front_idx[tid] = new_idx[tid]; front_score[tid] = new_score[tid]; }
        __syncthreads();
        if (tid == 0) {
            float c = 0.f;
            for (int f = 0; f < k; ++f) c = __fadd_rn(c, expf(front_score[f]));
            w.conf[b * D + d] = c;
            for (int s = 0; s < p.n_cp; ++s)
                if (p.checkpoint[s] == d && c < p.tau[s]) st = s;
        }
        __syncthreads();
        if (st >= 0) break;
    }
    if (tid == 0) {
        int out = st;
        if (out < 0 && d_hi == D - 1) out = p.n_cp;  // drafted every call: the dense stage
        w.state[b] = out;
    }
    if (tid < k) {
        w.front_idx[b * GRAFT_MAX_TOPK + tid] = front_idx[tid];
        w.front_score[b * GRAFT_MAX_TOPK + tid] = front_score[tid];
    }
}

struct MergeParams {
    int D, k, Kmax, n_cp;
    int checkpoint[GRAFT_MAX_CHECKPOINTS];
    int K_draft[GRAFT_MAX_CHECKPOINTS + 1];
    signed char tmpl_parent[GRAFT_MAX_KMAX];
};

constexpr int kMergeThreads = 512;

__global__ void __launch_bounds__(kMergeThreads)
draft_merge_kernel(MergeParams p, const int32_t* __restrict__ root_tok, const int32_t* __restrict__ L,
                   BuildWs w, int32_t* tree_tok, int32_t* tree_parent, int32_t* tree_depth,
                   int32_t* tree_pos, uint64_t* tree_mask, int32_t* stage_out, int32_t* status) {
    griddep_enter();
    const int b = blockIdx.x, tid = threadIdx.x;
    const int k = p.k, KK = k * k, Kmax = p.Kmax;
    extern __shared__ float sm_pool[];  // [P] scores
    __shared__ int node_of_kept[GRAFT_MAX_KMAX];
    __shared__ int kept_entry[GRAFT_MAX_KMAX];
    __shared__ int s_tok[GRAFT_MAX_KMAX], s_par[GRAFT_MAX_KMAX];

    int st = w.state[b];
    if (st < 0 || st > p.n_cp) st = p.n_cp;
    const int n_draft = p.K_draft[st];
    const int dmax = (st < p.n_cp) ? p.checkpoint[st] : p.D - 1;
    const int P = k + dmax * KK;
    // without retrieval K_draft_s = Kmax can exceed the pool: the whole pool is kept and the
    // remaining draft slots stay empty (token -1 under the root)
    const int keep = min(n_draft - 1, P);
    // pool entry e: call 0 holds entries [0, k); call d >= 1 holds [k + (d-1)k^2, k + d k^2)
    auto call_of = [&](int e) { return e < k ? 0 : 1 + (e - k) / KK; };
    auto idx_of = [&](int e) { return e < k ? e : (e - k) % KK; };
    auto gidx = [&](int e) { return ((size_t)b * p.D + call_of(e)) * KK + idx_of(e); };
    for (int e = tid; e < P; e += kMergeThreads) sm_pool[e] = w.pool_score[gidx(e)];
    __syncthreads();
    // keep the K_draft_s - 1 best entries by (score desc, depth asc, index asc):
    // entries are stored in (depth, index) order, so the tie-break is entry order
    for (int q = tid; q < GRAFT_MAX_KMAX; q += kMergeThreads) kept_entry[q] = -1;
    __syncthreads();
    for (int e = tid; e < P; e += kMergeThreads) {
        const float sc = sm_pool[e];
        int rank = 0;
        for (int e2 = 0; e2 < P && rank < keep; ++e2) {
            const float o = sm_pool[e2];
            rank += (o > sc) || (o == sc && e2 < e);
        }
        if (rank < keep) kept_entry[rank] = e;
    }
    __syncthreads();
    // scores are never NaN here, so the ranks are a permutation; a hole would mean a broken input
    if (tid < keep && (kept_entry[tid] < 0 || kept_entry[tid] >= P)) {
        flag_status(status, GRAFT_STATUS_TREE);
        kept_entry[tid] = 0;
    }
    __syncthreads();
    // every slot starts as a pad under the root, so the ancestor walk below ends even on a broken input;
    // draft slots past the kept pool are empty nodes
    if (tid < GRAFT_MAX_KMAX) {
        s_tok[tid] = (tid > keep && tid < n_draft) ? -1 : 0;
        s_par[tid] = tid == 0 ? -1 : 0;
    }
    // tree order among the kept: (depth asc, score desc, index asc)
    if (tid < keep) {
        const int e = kept_entry[tid];
        const int de = call_of(e);
        const float se = sm_pool[e];
        int pos = 0;
        for (int q = 0; q < keep; ++q) {
            const int e2 = kept_entry[q];
            const int d2 = call_of(e2);
            const float s2 = sm_pool[e2];
            pos += (d2 < de) || (d2 == de && (s2 > se || (s2 == se && e2 < e)));
        }
        node_of_kept[tid] = 1 + pos;
    }
    __syncthreads();
    if (tid < keep) {
        const int e = kept_entry[tid];
        const int node = node_of_kept[tid];
        const size_t g = gidx(e);
        s_tok[node] = w.pool_tok[g];
        const int d = call_of(e);
        int parent = 0;
        if (d >= 1) {
            const int pe = (d == 1 ? 0 : k + (d - 2) * KK) + w.pool_par[g];
            parent = -1;
            for (int q = 0; q < keep; ++q)
                if (kept_entry[q] == pe) parent = node_of_kept[q];
            // a parent precedes its child, which also keeps the ancestor walk below finite
            if (parent < 0 || parent >= node) { flag_status(status, GRAFT_STATUS_TREE); parent = 0; }
        }
        s_par[node] = parent;
    }
    if (tid == 0) { s_tok[0] = root_tok[b]; s_par[0] = -1; }
    const int n_ret = Kmax - n_draft;
    if (tid < n_ret) {
        const int t = w.ret[b * GRAFT_MAX_KMAX + tid];
        s_tok[n_draft + tid] = t >= 0 ? t : 0;
        const int tp = p.tmpl_parent[tid];
        s_par[n_draft + tid] = tp < 0 ? 0 : n_draft + tp;
    }
    __syncthreads();
    if (tid < Kmax) {
        uint64_t mask = 0;
        int depth = -1;
        for (int j = tid; j >= 0; j = s_par[j]) { mask |= 1ull << j; ++depth; }
        const size_t o = (size_t)b * Kmax + tid;
        tree_tok[o] = s_tok[tid];
        tree_parent[o] = s_par[tid];
        tree_depth[o] = depth;
        tree_pos[o] = L[b] + depth;
        tree_mask[o] = mask;
    }
    if (tid == 0) stage_out[b] = st;
}

struct TmplParams {
    int n, max_depth;
    signed char parent[GRAFT_MAX_KMAX];
    unsigned char rank[GRAFT_MAX_KMAX];
    unsigned char depth[GRAFT_MAX_KMAX];
};

__global__ void __launch_bounds__(GRAFT_MAX_KMAX)
retrieve_kernel(int V, int W, const int32_t* __restrict__ root_tok, const int32_t* __restrict__ M_succ,
                TmplParams tp, int32_t* __restrict__ out, int out_stride, int32_t* status) {
    griddep_enter();
    const int b = blockIdx.x, j = threadIdx.x;
    __shared__ int tok[GRAFT_MAX_KMAX];
    const int root = root_tok[b];
    const bool root_ok = root >= 0 && root < V;
    if (!root_ok && j == 0) flag_status(status, GRAFT_STATUS_TOKEN_RANGE);
    for (int lvl = 1; lvl <= tp.max_depth; ++lvl) {
        if (j < tp.n && tp.depth[j] == lvl) {
            const int par = tp.parent[j];
            const int ptok = par < 0 ? (root_ok ? root : -1) : tok[par];
            int t = -1;
            if (ptok >= 0) {
                t = __ldg(M_succ + (size_t)ptok * W + tp.rank[j]);
                if (t < -1 || t >= V) { flag_status(status, GRAFT_STATUS_TOKEN_RANGE); t = -1; }
            }
            tok[j] = t;
        }
        __syncthreads();
    }
    if (j < tp.n) out[(size_t)b * out_stride + j] = tok[j];
}

int row_splits(int V) {
    int S = (V + 8191) / 8192;
    return S < 1 ? 1 : (S > kMaxSplits ? kMaxSplits : S);
}

BuildWs carve_build(WsCarver& c, const GraftConfig* cfg, int B) {
    const int S = row_splits(cfg->V);
    const size_t rows = (size_t)B * cfg->D * cfg->k;
    BuildWs w;
    w.parts = c.take<RowPart>(rows * S);
    w.pool_score = c.take<float>(rows * cfg->k);
    w.pool_tok = c.take<int32_t>(rows * cfg->k);
    w.pool_par = c.take<int32_t>(rows * cfg->k);
    w.front_idx = c.take<int32_t>((size_t)B * GRAFT_MAX_TOPK);
    w.front_score = c.take<float>((size_t)B * GRAFT_MAX_TOPK);
    w.state = c.take<int32_t>(B);
    w.conf = c.take<float>((size_t)B * cfg->D);
    w.ret = c.take<int32_t>((size_t)B * GRAFT_MAX_KMAX);
    return w;
}

TmplParams make_tmpl(const GraftConfig* cfg) {
    TmplParams tp{};
    tp.n = cfg->n_tmpl;
    tp.max_depth = 0;
    for (int j = 0; j < cfg->n_tmpl; ++j) {
        tp.parent[j] = (signed char)cfg->tmpl_parent[j];
        tp.rank[j] = (unsigned char)cfg->tmpl_rank[j];
        const int d = cfg->tmpl_parent[j] < 0 ? 1 : tp.depth[cfg->tmpl_parent[j]] + 1;
        tp.depth[j] = (unsigned char)d;
        if (d > tp.max_depth) tp.max_depth = d;
    }
    return tp;
}

template <int KT>
void launch_rows(const float* logits, const GraftConfig* cfg, int B, int d_lo, int d_hi, int S, int chunk,
                 const int32_t* state, RowPart* parts, cudaStream_t st, int block) {
    dim3 grid(S, (d_hi - d_lo + 1) * cfg->k, B);
    launch_pdl(draft_rows_kernel<KT>, dim3(grid), dim3(kRowThreads), 0, st, logits, cfg->D, cfg->k, cfg->V, d_lo, S,
               chunk, state, parts, block);
    count_launches(1);
}

}  // namespace
}  // namespace graft

using namespace graft;

extern "C" int graft_build_tree_workspace_size(const GraftConfig* cfg, int B, size_t* bytes) {
    if (bytes == nullptr || B < 0) return GRAFT_ERR_INVALID_ARG;
    const int rc = graft_config_validate(cfg);
    if (rc != GRAFT_OK) return rc;
    WsCarver c(nullptr);
    carve_build(c, cfg, B);
    *bytes = c.bytes();
    return GRAFT_OK;
}

extern "C" int graft_retrieve(const GraftConfig* cfg, int B, const int32_t* root_tok, const int32_t* M_succ,
                              int32_t* ret_tok, int32_t* status, graft_stream_t stream) {
    const int rc = graft_config_validate(cfg);
    if (rc != GRAFT_OK) return rc;
    if (B < 0) return GRAFT_ERR_INVALID_ARG;
    if (B == 0 || cfg->n_tmpl == 0) return GRAFT_OK;
    if (root_tok == nullptr || M_succ == nullptr || ret_tok == nullptr) return GRAFT_ERR_INVALID_ARG;
    const TmplParams tp = make_tmpl(cfg);
    launch_pdl(retrieve_kernel, dim3(B), dim3(GRAFT_MAX_KMAX), 0, (cudaStream_t)stream, cfg->V, cfg->W, root_tok, M_succ, tp,
                                                                     ret_tok, cfg->n_tmpl, status);
    count_launches(1);
    return launch_status();
}

namespace {

int build_tree_impl(const GraftConfig* cfg, int B, const float* draft_logits, int block, const int32_t* root_tok,
                    const int32_t* M_succ, const int32_t* L, int32_t* tree_tok, int32_t* tree_parent,
                    int32_t* tree_depth, int32_t* tree_pos, uint64_t* tree_mask, int32_t* stage, int32_t* status,
                    void* ws, size_t ws_bytes, graft_stream_t stream) {
    const int rc = graft_config_validate(cfg);
    if (rc != GRAFT_OK) return rc;
    if (B < 0) return GRAFT_ERR_INVALID_ARG;
    if (B == 0) return GRAFT_OK;
    if (draft_logits == nullptr || root_tok == nullptr || M_succ == nullptr || L == nullptr ||
        tree_tok == nullptr || tree_parent == nullptr || tree_depth == nullptr || tree_pos == nullptr ||
        tree_mask == nullptr || stage == nullptr)
        return GRAFT_ERR_INVALID_ARG;
    if ((size_t)B * cfg->D * cfg->k > (size_t)65535 * 65535) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    WsCarver sizer(nullptr);
    carve_build(sizer, cfg, B);
    if (!ws_ok(ws, ws_bytes, sizer.bytes())) return GRAFT_ERR_WORKSPACE;
    WsCarver c(ws);
    BuildWs w = carve_build(c, cfg, B);
    cudaStream_t st = (cudaStream_t)stream;

    const int S = row_splits(cfg->V);
    int chunk = (cfg->V + S - 1) / S;
    chunk = (chunk + 3) & ~3;
    if (B > 65535) return GRAFT_ERR_UNSUPPORTED_SHAPE;

    const TmplParams tp = make_tmpl(cfg);
    if (cfg->n_tmpl > 0) {
        launch_pdl(retrieve_kernel, dim3(B), dim3(GRAFT_MAX_KMAX), 0, st, cfg->V, cfg->W, root_tok, M_succ, tp, w.ret,
                                                       GRAFT_MAX_KMAX, status);
        count_launches(1);
    }

    SelectParams sp{};
    sp.D = cfg->D;
    sp.k = cfg->k;
    sp.S = S;
    sp.n_cp = cfg->n_checkpoints;
    for (int s = 0; s < cfg->n_checkpoints; ++s) {
        sp.checkpoint[s] = cfg->checkpoint[s];
        sp.tau[s] = cfg->tau[s];
    }
    // groups of drafter calls ending at each checkpoint, then the tail
    int d_lo = 0;
    for (int g = 0; g <= cfg->n_checkpoints && d_lo < cfg->D; ++g) {
        const int d_hi = (g < cfg->n_checkpoints) ? cfg->checkpoint[g] : cfg->D - 1;
        const int32_t* gate = (d_lo == 0) ? nullptr : w.state;
        if (cfg->k <= 4) launch_rows<4>(draft_logits, cfg, B, d_lo, d_hi, S, chunk, gate, w.parts, st, block);
        else if (cfg->k <= 8) launch_rows<8>(draft_logits, cfg, B, d_lo, d_hi, S, chunk, gate, w.parts, st, block);
        else launch_rows<16>(draft_logits, cfg, B, d_lo, d_hi, S, chunk, gate, w.parts, st, block);
        launch_pdl(draft_select_kernel, dim3(B), dim3(kSelThreads), 0, st, sp, d_lo, d_hi, w);
        count_launches(1);
        d_lo = d_hi + 1;
    }

    MergeParams mp{};
    mp.D = cfg->D;
    mp.k = cfg->k;
    mp.Kmax = cfg->Kmax;
    mp.n_cp = cfg->n_checkpoints;
    for (int s = 0; s < cfg->n_checkpoints; ++s) mp.checkpoint[s] = cfg->checkpoint[s];
    for (int s = 0; s <= cfg->n_checkpoints; ++s) mp.K_draft[s] = cfg->K_draft[s];
    for (int j = 0; j < cfg->n_tmpl; ++j) mp.tmpl_parent[j] = (signed char)cfg->tmpl_parent[j];
    const int max_pool = cfg->k + (cfg->D - 1) * cfg->k * cfg->k;
    const size_t smem = (size_t)max_pool * sizeof(float);
    if (smem > 48 * 1024) {
        if (!cuda_ok(cudaFuncSetAttribute(draft_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
            return GRAFT_ERR_CUDA;
    }
    launch_pdl(draft_merge_kernel, dim3(B), dim3(kMergeThreads), smem, st, mp, root_tok, L, w, tree_tok, tree_parent, tree_depth,
                                                      tree_pos, tree_mask, stage, status);
    count_launches(1);
    return launch_status();
}

}  // namespace

extern "C" int graft_build_tree(const GraftConfig* cfg, int B, const float* draft_logits,
                                const int32_t* root_tok, const int32_t* M_succ, const int32_t* L,
                                int32_t* tree_tok, int32_t* tree_parent, int32_t* tree_depth,
                                int32_t* tree_pos, uint64_t* tree_mask, int32_t* stage,
                                int32_t* status, void* ws, size_t ws_bytes, graft_stream_t stream) {
    return build_tree_impl(cfg, B, draft_logits, 0, root_tok, M_succ, L, tree_tok, tree_parent, tree_depth, tree_pos,
                           tree_mask, stage, status, ws, ws_bytes, stream);
}

extern "C" int graft_build_tree_block(const GraftConfig* cfg, int B, const float* block_logits,
                                      const int32_t* root_tok, const int32_t* M_succ, const int32_t* L,
                                      int32_t* tree_tok, int32_t* tree_parent, int32_t* tree_depth,
                                      int32_t* tree_pos, uint64_t* tree_mask, int32_t* stage,
                                      int32_t* status, void* ws, size_t ws_bytes, graft_stream_t stream) {
    return build_tree_impl(cfg, B, block_logits, 1, root_tok, M_succ, L, tree_tok, tree_parent, tree_depth, tree_pos,
                           tree_mask, stage, status, ws, ws_bytes, stream);
}
