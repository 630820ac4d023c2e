// Stages 1-3 of the verify step: draft tree with dynamic-depth pruning,
// retrieval fill from M, and the hybrid merge.
//
// Graft article, step summary and method paragraph (first three points);
// architecture paragraph (checkpoints d0/d1/d5, Kmax = K_draft_s + K_ret_s,
// |T_s| = Kmax, per-stage template prefixes); Graft abstract
// ("prune-then-graft" fills the positions pruning opened).
//
// Kernel plan: ONE cooperative launch (every CTA resident), its phases
// separated by a grid barrier whose waits are bounded:
//   phase 0     the retrieval fill (one CTA per request, taken from the end of
//               the grid: level by level through M, independent of drafting)
//               and the row statistics of drafter-call group 0
//   for each checkpoint group g (the drafter calls between two checkpoints):
//     rows      every (row, split) item streams its share of one logit row
//               once: online log-sum-exp and a register top-k (HBM bound);
//               requests pruned at an earlier checkpoint are skipped, so rows
//               past the pruning point are never read
//     barrier
//     select    one CTA per request combines the splits, scores the children,
//               picks the next frontier, computes c_d and applies the gate at
//               the checkpoint; a request whose drafting ends here (pruned, or
//               its last call done) is merged at once by the same CTA: rerank
//               the pool, order the kept draft, append the stage's envelope
//               prefix, write parents, depths, positions and ancestor masks
//     barrier   (skipped after the last group; the launch ends early once no
//               request drafts on)
// A separate launch per stage would cost a kernel boundary each (ten of them
// with three checkpoints); the phases here cost one barrier each.
#include <climits>
#include <cmath>

#include "common.cuh"

namespace graft {
namespace {

// one block size for every phase: the row reductions, the per-request select and merge
constexpr int kThreads = 256;
constexpr int kMaxSplits = 32;
constexpr uint64_t kBarrierNs = 500000000ull;    // bound on one grid-barrier wait (phases take microseconds)

struct RowPart {
    float m;    // running max of the split
    float s;    // sum of exp(x - m) over the split
    float v[GRAFT_MAX_TOPK];
    int id[GRAFT_MAX_TOPK];
};

// (a, ia) strictly better than (b, ib): value desc, id asc; bitwise, so lanes never diverge on it
__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
    return (a > b) | ((a == b) & (ia < ib));
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
            const float nv = above ? v[j > 0 ? j - 1 : 0] : x;
            const int ni = above ? id[j > 0 ? j - 1 : 0] : i;
            v[j] = here ? nv : v[j];
            id[j] = here ? ni : id[j];
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
            const bool take = better(ov, oi, bv, bi) | ((ov == bv) & (oi == bi) & (ol < bl));
            bv = take ? ov : bv;
            bi = take ? oi : bi;
            bl = take ? ol : bl;
        }
        if (lane == 0) { out_v[r] = bv; out_id[r] = bi; }
        if (lane == bl) tk.pop();
    }
}

// Warp-wide bitonic sort of one (value, id) per lane into (value desc, id asc) order: lane j ends
// with the warp's j-th best.
__device__ __forceinline__ void warp_sort_desc(float& v, int& id) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, v, stride);
            const int oi = __shfl_xor_sync(0xffffffffu, id, stride);
            // in a best-first run the lower lane of a pair keeps the better entry, in a worst-first
            // run the worse one; the last merge (size 32) is best-first over the whole warp
            const bool keep_better = ((lane & stride) == 0) == ((lane & size) == 0);
            const bool take = keep_better ? better(ov, oi, v, id) : better(v, id, ov, oi);
            v = take ? ov : v;
            id = take ? oi : id;
        }
    }
}

constexpr int kRowVals = 32;  // values a thread holds at once (8 float4): a whole split of <= 8192

// Warp-wide log-sum-exp of (m, s) pairs (s = sum of exp(x - m)): the warp max, one rescale, a sum.
// Every lane ends with the warp's pair; an all -inf warp gives (-inf, 0).
__device__ __forceinline__ void warp_lse(float& m, float& s) {
    float wm = m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, off));
    float ws = m > -INFINITY ? s * __expf(m - wm) : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, off);
    m = wm;
    s = ws;
}

// One (row, split) item: the split's log-sum-exp (m, s) and its top-k by (value desc, id asc), NaN
// entries ignored, missing slots (-inf, INT_MAX), written to parts[(b, d, f) * S + s].  Every thread
// of the CTA calls it (it synchronises).
//
// Each thread holds its values in registers (one batch of kRowVals, or several for splits beyond
// kRowVals x kThreads values) and takes its own best entry and its (max, sum of exp) pair.  In each
// warp, the k-th best of the threads' own bests, tau_w, is a lower bound on the warp's k-th entry
// (the k threads above it hold k distinct entries at least as good), so the warp's top-k are among
// its entries at least as good as tau_w (all its non-NaN entries if fewer than k threads hold one).
// Those candidates, typically little more than k, are gathered one per lane and sorted: the first
// k lanes hold the warp's top-k.  The split's top-k are then the k best of the warps' top-k, found
// by ranking those NW x k entries against each other.  A warp with more than 32 candidates (rows of
// mass ties) sends the whole split down the per-thread insertion path instead.
template <int KT>
__device__ __forceinline__ void row_split_stats(const float* __restrict__ logits, int D, int k, int V, int S,
                                                int chunk, int block, int b, int d, int f, int s,
                                                RowPart* __restrict__ parts) {
    constexpr int NW = kThreads / 32;
    __shared__ float sm_m[NW], sm_s[NW];
    __shared__ float sm_v[NW][KT];
    __shared__ int sm_id[NW][KT];
    __shared__ float2 stage[NW][32];  // a warp's candidates (value, id as float bits)

    __syncthreads();  // the shared staging above is reused item after item
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the split's result goes to slot (b, d, f); block drafts read one row per depth, shared by
    // every frontier node of that depth
    const size_t row_id = ((size_t)b * D + d) * k + f;
    const size_t in_row = block ? (size_t)b * D + d : row_id;
    const float* row = logits + in_row * (size_t)V;
    const int lo = s * chunk;
    const int hi = min(V, lo + chunk);
    const bool vec = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
    constexpr int kBatch = kRowVals * kThreads;
    const int n_batch = (hi - lo + kBatch - 1) / kBatch;
    // value u of batch q of this thread: float4 groups of four adjacent ids (vector path) or one id
    // per thread stride (scalar path); ids past the split read as NaN, which every rule ignores
    auto id_of = [&](int q, int u) {
        return vec ? lo + q * kBatch + (u >> 2) * (4 * kThreads) + 4 * tid + (u & 3)
                   : lo + q * kBatch + u * kThreads + tid;
    };
    float x[kRowVals];
    auto load = [&](int q) {
        if (vec) {
#pragma unroll
            for (int u4 = 0; u4 < kRowVals / 4; ++u4) {
                const int i = id_of(q, 4 * u4);
                float4 w = make_float4(NAN, NAN, NAN, NAN);
                if (i < hi) w = __ldcs(reinterpret_cast<const float4*>(row + i));
                x[4 * u4] = w.x;
                x[4 * u4 + 1] = w.y;
                x[4 * u4 + 2] = w.z;
                x[4 * u4 + 3] = w.w;
            }
        } else {
#pragma unroll
            for (int u = 0; u < kRowVals; ++u) {
                const int i = id_of(q, u);
                x[u] = i < hi ? __ldcs(row + i) : NAN;
            }
        }
    };

    // this thread's best entry and (max, sum of exp(x - max)) over its values
    float bv = -INFINITY, m = -INFINITY, sum = 0.f;
    int bi = INT_MAX;
    for (int q = 0; q < n_batch; ++q) {
        load(q);
        float qm = -INFINITY;
#pragma unroll
        for (int u = 0; u < kRowVals; ++u) {
            const bool bt = better(x[u], id_of(q, u), bv, bi);
            bv = bt ? x[u] : bv;
            bi = bt ? id_of(q, u) : bi;
            qm = fmaxf(qm, x[u]);
        }
        float qs[4] = {0.f, 0.f, 0.f, 0.f};
        if (qm > -INFINITY) {
#pragma unroll
            for (int u = 0; u < kRowVals; ++u) qs[u & 3] += x[u] > -INFINITY ? __expf(x[u] - qm) : 0.f;
        }
        lse_merge(m, sum, qm, (qs[0] + qs[1]) + (qs[2] + qs[3]));
    }
    warp_lse(m, sum);
    if (lane == 0) { sm_m[warp] = m; sm_s[warp] = sum; }

    // tau_w: the warp's k-th best thread best (the sentinel (-inf, INT_MAX) passes every entry)
    float tv = bv;
    int ti = bi;
    warp_sort_desc(tv, ti);
    tv = __shfl_sync(0xffffffffu, tv, k - 1);
    ti = __shfl_sync(0xffffffffu, ti, k - 1);
    // gather the warp's candidates, one per lane
    int cnt = 0;
    for (int q = 0; q < n_batch; ++q) {
        if (n_batch > 1) load(q);
#pragma unroll
        for (int u = 0; u < kRowVals; ++u) {
            const int i = id_of(q, u);
            const bool pass = better(x[u], i, tv, ti) | ((x[u] == tv) & (i == ti));
            const unsigned bal = __ballot_sync(0xffffffffu, pass);
            if (bal != 0u) {
                const int pos = cnt + __popc(bal & ((1u << lane) - 1u));
                if (pass && pos < 32) stage[warp][pos] = make_float2(x[u], __int_as_float(i));
                cnt += __popc(bal);
            }
        }
    }
    __syncwarp();
    float cv = -INFINITY;
    int ci = INT_MAX;
    if (lane < min(cnt, 32)) {
        const float2 e = stage[warp][lane];
        cv = e.x;
        ci = __float_as_int(e.y);
    }
    warp_sort_desc(cv, ci);
    if (lane < k) { sm_v[warp][lane] = cv; sm_id[warp][lane] = ci; }
    const bool fallback = __syncthreads_or(cnt > 32);
    RowPart* out = parts + row_id * S + s;
    if (!fallback) {
        // rank the NW x k warp winners: real entries have distinct ids; equal sentinels (-inf,
        // INT_MAX) are ordered by their slot, so the ranks are a permutation and the first k slots
        // are each written once (by a sentinel where the split holds fewer than k entries)
        if (tid < NW * k) {
            const int w0 = tid / k, j0 = tid % k;
            const int me = w0 * KT + j0;
            const float v = sm_v[w0][j0];
            const int id = sm_id[w0][j0];
            int rank = 0;
            for (int w = 0; w < NW; ++w) {
#pragma unroll
                for (int j = 0; j < KT; ++j) {
                    const float ov = sm_v[w][j];
                    const int oi = sm_id[w][j];
                    rank += (j < k) & (better(ov, oi, v, id) | ((ov == v) & (oi == id) & (w * KT + j < me)));
                }
            }
            if (rank < k) { out->v[rank] = v; out->id[rank] = id; }
        }
    } else {
        // per-thread insertion top-k over the thread's values, then two warp tournaments
        __syncthreads();  // every warp has read its winners' slots
        TopK<KT> tk;
        tk.init();
        for (int q = 0; q < n_batch; ++q) {
            if (n_batch > 1) load(q);
#pragma unroll
            for (int u = 0; u < kRowVals; ++u) tk.offer(x[u], id_of(q, u));
        }
        warp_topk<KT>(tk, sm_v[warp], sm_id[warp]);
        __syncthreads();
        if (warp == 0) {
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
            if (lane < k) { out->v[lane] = fin_v[lane]; out->id[lane] = fin_id[lane]; }
        }
    }
    if (warp == 0) {
        m = lane < NW ? sm_m[lane] : -INFINITY;
        sum = lane < NW ? sm_s[lane] : 0.f;
        warp_lse(m, sum);
        if (lane == 0) { out->m = m; out->s = sum; }
    }
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
    uint32_t* bar;        // grid barrier word (low 31 bits zero between launches)
    int32_t* active;      // [n_checkpoints + 1] requests still drafting after each group's select
};

// Drafter calls d_lo..d_hi of request b (one CTA, every thread calls it): returns the request's state
// afterwards, -1 while it drafts on, else its stage (pruned at checkpoint s, or n_cp after the last call).
template <int KT>
__device__ __forceinline__ int select_group(const SelectParams& p, int d_lo, int d_hi, const BuildWs& w, int b) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NW = kThreads / 32;
    const int k = p.k, D = p.D, S = p.S;
    const int KK = k * k;

    __shared__ float lse_s[GRAFT_MAX_TOPK];
    __shared__ float top_v[GRAFT_MAX_TOPK][GRAFT_MAX_TOPK];
    __shared__ int top_id[GRAFT_MAX_TOPK][GRAFT_MAX_TOPK];
    __shared__ float cand_score[GRAFT_MAX_TOPK * GRAFT_MAX_TOPK];
    __shared__ int front_idx[GRAFT_MAX_TOPK];
    __shared__ float front_score[GRAFT_MAX_TOPK];
    __shared__ float2 sel_stage[NW][32];
    __shared__ int new_idx[GRAFT_MAX_TOPK];
    __shared__ float new_score[GRAFT_MAX_TOPK];
    __shared__ int st;

    __syncthreads();  // the shared state below is reused request after request
    if (d_lo > 0 && tid < k) {
        front_idx[tid] = __ldcg(w.front_idx + b * GRAFT_MAX_TOPK + tid);
        front_score[tid] = __ldcg(w.front_score + b * GRAFT_MAX_TOPK + tid);
    }
    if (tid == 0) st = -1;
    __syncthreads();

    for (int d = d_lo; d <= d_hi; ++d) {
        const int np = (d == 0) ? 1 : k;
        // combine the splits of every parent row of this call
        for (int f = warp; f < np; f += NW) {
            const RowPart* rp = w.parts + (((size_t)b * D + d) * k + f) * S;
            // S <= 32 splits, one per lane: its (max, sum) and its sorted list, loaded together
            float m = -INFINITY, sum = 0.f;
            TopK<KT> tl;
            tl.init();
            if (lane < S) {
#pragma unroll
                for (int j = 0; j < KT; ++j)
                    if (j < k) { tl.v[j] = __ldcg(&rp[lane].v[j]); tl.id[j] = __ldcg(&rp[lane].id[j]); }
                lse_merge(m, sum, __ldcg(&rp[lane].m), __ldcg(&rp[lane].s));
            }
            warp_lse(m, sum);
            // The k-th best list head tau is a lower bound on the union's k-th entry, so the union's
            // top-k lie in the lists' prefixes at least as good as tau; with S >= k heads and at most
            // 32 such entries they are gathered one per lane and sorted, else a k-round tournament.
            bool done = false;
            if (S >= k) {
                float hv = tl.v[0];
                int hid = tl.id[0];
                warp_sort_desc(hv, hid);
                const float tv = __shfl_sync(0xffffffffu, hv, k - 1);
                const int ti = __shfl_sync(0xffffffffu, hid, k - 1);
                int c = 0;
#pragma unroll
                for (int j = 0; j < KT; ++j)
                    c += (j < k) & (better(tl.v[j], tl.id[j], tv, ti) | ((tl.v[j] == tv) & (tl.id[j] == ti)));
                int incl = c;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int o = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += o;
                }
                const int total = __shfl_sync(0xffffffffu, incl, 31);
                if (total <= 32) {
#pragma unroll
                    for (int j = 0; j < KT; ++j)
                        if (j < c) sel_stage[warp][incl - c + j] = make_float2(tl.v[j], __int_as_float(tl.id[j]));
                    __syncwarp();
                    float cv = -INFINITY;
                    int ci = INT_MAX;
                    if (lane < total) {
                        const float2 e = sel_stage[warp][lane];
                        cv = e.x;
                        ci = __float_as_int(e.y);
                    }
                    __syncwarp();
                    warp_sort_desc(cv, ci);
                    if (lane < k) { top_v[f][lane] = cv; top_id[f][lane] = ci; }
                    done = true;
                }
            }
            if (!done) warp_topk<KT>(tl, top_v[f], top_id[f]);  // k-round tournament over the lists
            if (lane == 0) lse_s[f] = m + logf(sum);
        }
        __syncthreads();
        // score every child: parent score + (logit - lse), single float32 operations
        const int nc = np * k;
        for (int c = tid; c < nc; c += kThreads) {
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
        for (int c = tid; c < nc; c += kThreads) {
            const float sc = cand_score[c];
            int rank = 0;
            for (int c0 = 0; c0 < nc; c0 += 8) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int c2 = c0 + u;
                    if (c2 < nc) {
                        const float o = cand_score[c2];
                        rank += (o > sc) | ((o == sc) & (c2 < c));
                    }
                }
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
    int out = st;
    if (out < 0 && d_hi == D - 1) out = p.n_cp;  // drafted every call: the dense stage
    if (tid == 0) w.state[b] = out;
    if (tid < k) {
        w.front_idx[b * GRAFT_MAX_TOPK + tid] = front_idx[tid];
        w.front_score[b * GRAFT_MAX_TOPK + tid] = front_score[tid];
    }
    return out;
}

struct MergeParams {
    int D, k, Kmax, n_cp;
    int max_pool;  // k + (D - 1) k^2: the pool of the dense stage (shared-memory staging size)
    int checkpoint[GRAFT_MAX_CHECKPOINTS];
    int K_draft[GRAFT_MAX_CHECKPOINTS + 1];
    signed char tmpl_parent[GRAFT_MAX_KMAX];
};

struct TreeOut {
    const int32_t* root_tok;
    const int32_t* L;
    int32_t *tok, *parent, *depth, *pos;
    uint64_t* mask;
    int32_t* stage;
    int32_t* status;
};

// The tree of request b at stage st (one CTA, every thread calls it).  The pool's scores, tokens
// and parent indices are staged in dynamic shared memory (3 x max_pool words), loaded in one
// round trip together with the envelope tokens, the root token and the cache length.
__device__ __forceinline__ void merge_request(const MergeParams& p, const BuildWs& w, const TreeOut& o, int b, int st) {
    constexpr int kMergeThreads = kThreads;
    const int tid = threadIdx.x;
    const int k = p.k, KK = k * k, Kmax = p.Kmax;
    extern __shared__ float sm_pool[];  // [max_pool] scores, then [max_pool] tokens and parent indices
    int* sm_ptok = reinterpret_cast<int*>(sm_pool + p.max_pool);
    int* sm_ppar = sm_ptok + p.max_pool;
    __shared__ int node_of_kept[GRAFT_MAX_KMAX];
    __shared__ int kept_entry[GRAFT_MAX_KMAX];
    __shared__ int s_tok[GRAFT_MAX_KMAX], s_par[GRAFT_MAX_KMAX];
    __shared__ int s_ret[GRAFT_MAX_KMAX];
    __shared__ int s_root, s_L;

    __syncthreads();  // the shared state below is reused request after request
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
    const int n_ret = Kmax - n_draft;
    for (int e = tid; e < P; e += kMergeThreads) {
        const size_t g = gidx(e);
        sm_pool[e] = __ldcg(w.pool_score + g);
        sm_ptok[e] = __ldcg(w.pool_tok + g);
        sm_ppar[e] = __ldcg(w.pool_par + g);
    }
    if (tid < n_ret) s_ret[tid] = __ldcg(w.ret + b * GRAFT_MAX_KMAX + tid);
    if (tid == 0) { s_root = o.root_tok[b]; s_L = o.L[b]; }
    __syncthreads();
    // keep the K_draft_s - 1 best entries by (score desc, depth asc, index asc):
    // entries are stored in (depth, index) order, so the tie-break is entry order
    for (int q = tid; q < GRAFT_MAX_KMAX; q += kMergeThreads) kept_entry[q] = -1;
    __syncthreads();
    for (int e = tid; e < P; e += kMergeThreads) {
        const float sc = sm_pool[e];
        int rank = 0;
        for (int e0 = 0; e0 < P && rank < keep; e0 += 8) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e2 = e0 + u;
                if (e2 < P) {
                    const float o = sm_pool[e2];
                    rank += (o > sc) | ((o == sc) & (e2 < e));
                }
            }
        }
        if (rank < keep) kept_entry[rank] = e;
    }
    __syncthreads();
    // scores are never NaN here, so the ranks are a permutation; a hole would mean a broken input
    if (tid < keep && (kept_entry[tid] < 0 || kept_entry[tid] >= P)) {
        flag_status(o.status, GRAFT_STATUS_TREE);
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
#pragma unroll 4
        for (int q = 0; q < keep; ++q) {
            const int e2 = kept_entry[q];
            const int d2 = call_of(e2);
            const float s2 = sm_pool[e2];
            pos += (d2 < de) | ((d2 == de) & ((s2 > se) | ((s2 == se) & (e2 < e))));
        }
        node_of_kept[tid] = 1 + pos;
    }
    __syncthreads();
    if (tid < keep) {
        const int e = kept_entry[tid];
        const int node = node_of_kept[tid];
        s_tok[node] = sm_ptok[e];
        const int d = call_of(e);
        int parent = 0;
        if (d >= 1) {
            const int pe = (d == 1 ? 0 : k + (d - 2) * KK) + sm_ppar[e];
            parent = -1;
            for (int q = 0; q < keep; ++q)
                if (kept_entry[q] == pe) parent = node_of_kept[q];
            // a parent precedes its child, which also keeps the ancestor walk below finite
            if (parent < 0 || parent >= node) { flag_status(o.status, GRAFT_STATUS_TREE); parent = 0; }
        }
        s_par[node] = parent;
    }
    if (tid == 0) { s_tok[0] = s_root; s_par[0] = -1; }
    if (tid < n_ret) {
        const int t = s_ret[tid];
        s_tok[n_draft + tid] = t >= 0 ? t : 0;
        const int tp = p.tmpl_parent[tid];
        s_par[n_draft + tid] = tp < 0 ? 0 : n_draft + tp;
    }
    __syncthreads();
    if (tid < Kmax) {
        uint64_t mask = 0;
        int depth = -1;
        for (int j = tid; j >= 0; j = s_par[j]) { mask |= 1ull << j; ++depth; }
        const size_t i = (size_t)b * Kmax + tid;
        o.tok[i] = s_tok[tid];
        o.parent[i] = s_par[tid];
        o.depth[i] = depth;
        o.pos[i] = s_L + depth;
        o.mask[i] = mask;
    }
    if (tid == 0) o.stage[b] = st;
}

struct TmplParams {
    int n, max_depth;
    signed char parent[GRAFT_MAX_KMAX];
    unsigned char rank[GRAFT_MAX_KMAX];
    unsigned char depth[GRAFT_MAX_KMAX];
};

// The envelope tokens of request b (threads 0..n-1 hold the template's nodes; every thread of the CTA
// calls it, it synchronises level by level).
__device__ __forceinline__ void retrieve_request(int V, int W, const int32_t* __restrict__ root_tok,
                                 const int32_t* __restrict__ M_succ, const TmplParams& tp,
                                 int32_t* __restrict__ out, int out_stride, int32_t* status, int b) {
    const int j = threadIdx.x;
    __shared__ int tok[GRAFT_MAX_KMAX];
    __syncthreads();  // reused request after request
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

__global__ void __launch_bounds__(GRAFT_MAX_KMAX)
retrieve_kernel(int V, int W, const int32_t* __restrict__ root_tok, const int32_t* __restrict__ M_succ,
                TmplParams tp, int32_t* __restrict__ out, int out_stride, int32_t* status) {
    griddep_enter();
    retrieve_request(V, W, root_tok, M_succ, tp, out, out_stride, status, blockIdx.x);
}

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Grid-wide barrier of a cooperative launch on one 32-bit word: every CTA adds 1 except CTA 0,
// which adds 2^31 - (gridDim.x - 1), so one barrier adds exactly 2^31: the top bit flips when the
// last CTA arrives and the low 31 bits are back at zero.  The word's low bits must start at zero
// (the workspace is zero-filled once; every completed call leaves them at zero).  The arrival is a
// release and the polling an acquire at GPU scope, so writes before the barrier are visible after
// it.  A wait gives up after kBarrierNs: the CTA flags GRAFT_STATUS_TIMEOUT and the function
// returns false (the CTA then ends; so do the others, at their next bounded wait).
__device__ __forceinline__ bool grid_barrier(uint32_t* bar, int32_t* status) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        const uint32_t add = blockIdx.x == 0 ? 0x80000000u - (gridDim.x - 1) : 1u;
        uint32_t old;
        asm volatile("atom.add.release.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(bar), "r"(add) : "memory");
        // during a barrier the low bits are below gridDim.x, or at least 2^31 - (gridDim.x - 1) once
        // CTA 0 has arrived: anything between means the word was not zeroed
        const uint32_t low = old & 0x7fffffffu;
        if (low >= gridDim.x && low < 0x80000000u - (gridDim.x - 1)) flag_status(status, GRAFT_STATUS_WORKSPACE);
        const uint64_t t0 = now_ns();
        for (;;) {
            uint32_t cur;
            asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(cur) : "l"(bar) : "memory");
            if ((cur ^ old) & 0x80000000u) break;
            if (now_ns() - t0 > kBarrierNs) {
                flag_status(status, GRAFT_STATUS_TIMEOUT);
                ok = 0;
                break;
            }
            __nanosleep(20);
        }
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

struct BuildArgs {
    const float* logits;
    int block;  // 1: one logit row per depth (block drafter), shared by the depth's frontier
    int B, V, W, S, chunk, n_tmpl, n_groups;
    int grp_lo[GRAFT_MAX_CHECKPOINTS + 1], grp_hi[GRAFT_MAX_CHECKPOINTS + 1];
    const int32_t* M_succ;
    SelectParams sp;
    MergeParams mp;
    TmplParams tp;
    BuildWs w;
    TreeOut o;
};

// Rows of drafter calls d_lo..d_hi: call 0 has one row (the root's), later calls k rows each.
__device__ __forceinline__ int group_rows(int d_lo, int d_hi, int k) {
    return (d_hi - d_lo + 1) * k - (d_lo == 0 ? k - 1 : 0);
}

template <int KT>
__global__ void __launch_bounds__(kThreads, 2) build_tree_kernel(BuildArgs a) {
    griddep_enter();
    const int nb = gridDim.x, c = blockIdx.x;
    const int k = a.sp.k, D = a.sp.D, S = a.S;
    // phase 0: the retrieval fill, from the last CTA down (the first CTAs take the first row items)
    if (a.n_tmpl > 0)
        for (int b = nb - 1 - c; b < a.B; b += nb)
            retrieve_request(a.V, a.W, a.o.root_tok, a.M_succ, a.tp, a.w.ret, GRAFT_MAX_KMAX, a.o.status, b);
    if (c == 0 && threadIdx.x < a.n_groups) a.w.active[threadIdx.x] = 0;  // read after group 0's barriers
    for (int g = 0; g < a.n_groups; ++g) {
        const int d_lo = a.grp_lo[g], d_hi = a.grp_hi[g];
        const int nr = group_rows(d_lo, d_hi, k);
        const long long items = (long long)a.B * nr * S;
        for (long long i = c; i < items; i += nb) {
            const int s = (int)(i % S);
            const int r = (int)((i / S) % nr);
            const int b = (int)(i / ((long long)S * nr));
            if (g > 0 && __ldcg(a.w.state + b) != -1) continue;  // pruned at an earlier checkpoint
            int d, f;
            if (d_lo == 0) { d = r == 0 ? 0 : 1 + (r - 1) / k; f = r == 0 ? 0 : (r - 1) % k; }
            else { d = d_lo + r / k; f = r % k; }
            row_split_stats<KT>(a.logits, D, k, a.V, S, a.chunk, a.block, b, d, f, s, a.w.parts);
        }
        if (!grid_barrier(a.w.bar, a.o.status)) return;
        for (int b = c; b < a.B; b += nb) {
            if (g > 0 && __ldcg(a.w.state + b) != -1) continue;
            const int st = select_group<KT>(a.sp, d_lo, d_hi, a.w, b);
            if (st >= 0) merge_request(a.mp, a.w, a.o, b, st);
            else if (threadIdx.x == 0) atomicAdd(a.w.active + g, 1);
        }
        if (g == a.n_groups - 1) break;  // every request has ended
        if (!grid_barrier(a.w.bar, a.o.status)) return;
        if (__ldcg(a.w.active + g) == 0) break;
    }
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
    w.bar = c.take<uint32_t>(1);
    w.active = c.take<int32_t>(GRAFT_MAX_CHECKPOINTS + 1);
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

// CTAs of the cooperative launch: one per SM while the first group's row items (always read) do
// not fill the SMs, else every CTA the device holds at once (occupancy x SMs, more loads in flight);
// never more than the largest phase has work items.  The occupancy is cached per device ordinal.
template <int KT>
int coop_grid(size_t smem, long long first_items, long long max_items, int* grid) {
    static int per_sm[64] = {0};
    static size_t per_sm_smem[64] = {0};
    int dev = 0;
    if (!cuda_ok(cudaGetDevice(&dev))) return GRAFT_ERR_CUDA;
    if (dev < 0 || dev >= 64) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    if (per_sm[dev] == 0 || per_sm_smem[dev] != smem) {
        int n = 0;
        if (!cuda_ok(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, build_tree_kernel<KT>, kThreads, smem)))
            return GRAFT_ERR_CUDA;
        if (n < 1) return GRAFT_ERR_UNSUPPORTED_SHAPE;
        per_sm[dev] = n;
        per_sm_smem[dev] = smem;
    }
    const long long sms = device_sm_count();
    if (sms < 1) return GRAFT_ERR_CUDA;
    const long long cap = first_items < sms ? sms : (long long)per_sm[dev] * sms;
    *grid = (int)(max_items < 1 ? 1 : (max_items < cap ? max_items : cap));
    return GRAFT_OK;
}

template <int KT>
int launch_build(BuildArgs& a, size_t smem, long long first_items, long long max_items, cudaStream_t st) {
    // the kernel's static shared memory is below 16 KB: past 32 KB of dynamic staging, opt in
    if (smem > 32 * 1024 &&
        !cuda_ok(cudaFuncSetAttribute(build_tree_kernel<KT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
        return GRAFT_ERR_CUDA;
    int grid = 0;
    const int rc = coop_grid<KT>(smem, first_items, max_items, &grid);
    if (rc != GRAFT_OK) return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident: the phases meet at grid barriers
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!cuda_ok(cudaLaunchKernelEx(&cfg, build_tree_kernel<KT>, a))) return GRAFT_ERR_CUDA;
    count_launches(1);
    return GRAFT_OK;
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

    BuildArgs a{};
    a.logits = draft_logits;
    a.block = block;
    a.B = B;
    a.V = cfg->V;
    a.W = cfg->W;
    a.S = row_splits(cfg->V);
    a.chunk = ((cfg->V + a.S - 1) / a.S + 3) & ~3;
    a.n_tmpl = cfg->n_tmpl;
    a.M_succ = M_succ;
    a.tp = make_tmpl(cfg);
    a.w = w;
    a.o = TreeOut{root_tok, L, tree_tok, tree_parent, tree_depth, tree_pos, tree_mask, stage, status};

    SelectParams& sp = a.sp;
    sp.D = cfg->D;
    sp.k = cfg->k;
    sp.S = a.S;
    sp.n_cp = cfg->n_checkpoints;
    for (int s = 0; s < cfg->n_checkpoints; ++s) {
        sp.checkpoint[s] = cfg->checkpoint[s];
        sp.tau[s] = cfg->tau[s];
    }
    // groups of drafter calls ending at each checkpoint, then the tail
    long long max_items = B, first_items = 0;
    int d_lo = 0;
    for (int g = 0; g <= cfg->n_checkpoints && d_lo < cfg->D; ++g) {
        const int d_hi = (g < cfg->n_checkpoints) ? cfg->checkpoint[g] : cfg->D - 1;
        a.grp_lo[a.n_groups] = d_lo;
        a.grp_hi[a.n_groups] = d_hi;
        ++a.n_groups;
        const long long rows = (long long)(d_hi - d_lo + 1) * cfg->k - (d_lo == 0 ? cfg->k - 1 : 0);
        if ((long long)B * rows * a.S > max_items) max_items = (long long)B * rows * a.S;
        if (g == 0) first_items = (long long)B * rows * a.S;
        d_lo = d_hi + 1;
    }

    MergeParams& mp = a.mp;
    mp.D = cfg->D;
    mp.k = cfg->k;
    mp.Kmax = cfg->Kmax;
    mp.n_cp = cfg->n_checkpoints;
    for (int s = 0; s < cfg->n_checkpoints; ++s) mp.checkpoint[s] = cfg->checkpoint[s];
    for (int s = 0; s <= cfg->n_checkpoints; ++s) mp.K_draft[s] = cfg->K_draft[s];
    for (int j = 0; j < cfg->n_tmpl; ++j) mp.tmpl_parent[j] = (signed char)cfg->tmpl_parent[j];
    const int max_pool = cfg->k + (cfg->D - 1) * cfg->k * cfg->k;
    mp.max_pool = max_pool;
    const size_t smem = 3 * (size_t)max_pool * sizeof(float);

    int rc2;
    if (cfg->k <= 4) rc2 = launch_build<4>(a, smem, first_items, max_items, st);
    else if (cfg->k <= 8) rc2 = launch_build<8>(a, smem, first_items, max_items, st);
    else rc2 = launch_build<16>(a, smem, first_items, max_items, st);
    if (rc2 != GRAFT_OK) return rc2;
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
