// Host-side configuration, status strings and device queries of libgraft.
//
// The budget split and the retrieval envelope implement the Graft article's
// method paragraph (first and second points) and architecture paragraph:
// Kmax = K_draft_s + K_ret_s per pruning stage, more retrieval at smaller s,
// and per-stage templates that are prefixes of one envelope.  The pages give
// no numbers for either, so the library uses the readings documented in
// graft.h (graft_config_init).
#include <algorithm>
#include <atomic>
#include <cstring>
#include <vector>

#include "common.cuh"

namespace graft {

static std::atomic<unsigned long long> g_launches{0};

void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

static thread_local cudaError_t g_last_cuda_error = cudaSuccess;

void note_cuda_error(cudaError_t e) { g_last_cuda_error = e; }

int device_sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;
    }
    return cached[dev];
}

namespace {

struct RankPath {
    int len;
    int r[GRAFT_MAX_DEPTH];
    long long prod;
};

// Orders envelope nodes by (product of (rank + 1), length, lexicographic).
bool path_before(const RankPath& a, const RankPath& b) {
    if (a.prod != b.prod) return a.prod < b.prod;
    if (a.len != b.len) return a.len < b.len;
    for (int i = 0; i < a.len; ++i)
        if (a.r[i] != b.r[i]) return a.r[i] < b.r[i];
    return false;
}

void collect(RankPath& cur, int D, int W, long long bound, std::vector<RankPath>& out, size_t cap) {
    if (cur.len == D || out.size() > cap) return;
    for (int r = 0; r < W; ++r) {
        long long p = cur.prod * (r + 1);
        if (p > bound) break;
        RankPath next = cur;
        next.r[next.len++] = r;
        next.prod = p;
        out.push_back(next);
        collect(next, D, W, bound, out, cap);
    }
}

bool same_prefix(const RankPath& parent, const RankPath& child) {
    if (parent.len + 1 != child.len) return false;
    for (int i = 0; i < parent.len; ++i)
        if (parent.r[i] != child.r[i]) return false;
    return true;
}

int build_envelope(int D, int W, int n, int32_t* parent, int32_t* rank) {
    if (n == 0) return GRAFT_OK;
    // total number of rank paths, saturating
    long long total = 0, pw = 1;
    for (int m = 1; m <= D && total < n; ++m) {
        pw = std::min<long long>(pw * W, 1LL << 40);
        total += pw;
    }
    if (total < n) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    std::vector<RankPath> paths;
    for (long long bound = 1;; ++bound) {
        paths.clear();
        RankPath root{};
        root.len = 0;
        root.prod = 1;
        // cap keeps the search small: once the bound admits n paths we stop growing it
        collect(root, D, W, bound, paths, 1u << 20);
        if ((int)paths.size() >= n) break;
    }
    std::sort(paths.begin(), paths.end(), path_before);
    for (int j = 0; j < n; ++j) {
        rank[j] = paths[j].r[paths[j].len - 1];
        parent[j] = -1;
        if (paths[j].len > 1) {
            for (int q = 0; q < j; ++q)
                if (same_prefix(paths[q], paths[j])) { parent[j] = q; break; }
            if (parent[j] < 0) return GRAFT_ERR_INVALID_ARG;  // not ancestor-closed (cannot happen)
        }
    }
    return GRAFT_OK;
}

}  // namespace
}  // namespace graft

extern "C" int graft_config_validate(const GraftConfig* c) {
    if (c == nullptr) return GRAFT_ERR_INVALID_ARG;
    if (c->Kmax < 1 || c->Kmax > GRAFT_MAX_KMAX) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    if (c->D < 1 || c->D > GRAFT_MAX_DEPTH) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    if (c->k < 1 || c->k > GRAFT_MAX_TOPK) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    if (c->W < 1 || c->W > GRAFT_MAX_W) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    if (c->V < 1 || c->V < c->k) return GRAFT_ERR_INVALID_ARG;
    if (c->n_checkpoints < 0 || c->n_checkpoints > GRAFT_MAX_CHECKPOINTS) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    int prev = -1;
    for (int s = 0; s < c->n_checkpoints; ++s) {
        if (c->checkpoint[s] <= prev || c->checkpoint[s] >= c->D) return GRAFT_ERR_INVALID_ARG;
        prev = c->checkpoint[s];
    }
    if (c->K_draft[c->n_checkpoints] != c->Kmax) return GRAFT_ERR_INVALID_ARG;
    const long long full_pool = c->k + (long long)(c->D - 1) * c->k * c->k;
    if (full_pool < c->Kmax - 1) return GRAFT_ERR_INVALID_ARG;
    // K_draft[s] - 1 may exceed the stage's pool (k + d_s k^2 candidates): the pool is then kept
    // whole and the remaining draft slots are empty nodes (graft_config_no_retrieval)
    int need_tmpl = 0;
    for (int s = 0; s <= c->n_checkpoints; ++s) {
        const int kd = c->K_draft[s];
        if (kd < 1 || kd > c->Kmax) return GRAFT_ERR_INVALID_ARG;
        need_tmpl = std::max(need_tmpl, c->Kmax - kd);
    }
    if (c->n_tmpl < need_tmpl || c->n_tmpl > GRAFT_MAX_KMAX) return GRAFT_ERR_INVALID_ARG;
    for (int j = 0; j < c->n_tmpl; ++j) {
        if (c->tmpl_parent[j] < -1 || c->tmpl_parent[j] >= j) return GRAFT_ERR_INVALID_ARG;
        if (c->tmpl_rank[j] < 0 || c->tmpl_rank[j] >= c->W) return GRAFT_ERR_INVALID_ARG;
    }
    // a template node may not be deeper than the tree can index (depth <= D)
    int depth[GRAFT_MAX_KMAX];
    for (int j = 0; j < c->n_tmpl; ++j) {
        depth[j] = c->tmpl_parent[j] < 0 ? 1 : depth[c->tmpl_parent[j]] + 1;
        if (depth[j] > GRAFT_MAX_KMAX) return GRAFT_ERR_INVALID_ARG;
    }
    return GRAFT_OK;
}

extern "C" int graft_config_init(GraftConfig* cfg, int Kmax, int D, int k, int V, int W,
                                 int n_checkpoints, const int32_t* checkpoints, const float* tau) {
    if (cfg == nullptr || n_checkpoints < 0 || (n_checkpoints > 0 && (checkpoints == nullptr || tau == nullptr)))
        return GRAFT_ERR_INVALID_ARG;
    if (Kmax < 1 || Kmax > GRAFT_MAX_KMAX || D < 1 || D > GRAFT_MAX_DEPTH || k < 1 ||
        k > GRAFT_MAX_TOPK || W < 1 || W > GRAFT_MAX_W)
        return GRAFT_ERR_UNSUPPORTED_SHAPE;
    if (V < k) return GRAFT_ERR_INVALID_ARG;
    std::memset(cfg, 0, sizeof(*cfg));
    cfg->Kmax = Kmax;
    cfg->D = D;
    cfg->k = k;
    cfg->V = V;
    cfg->W = W;
    int ncp = 0;
    int prev = -1;
    for (int s = 0; s < n_checkpoints; ++s) {
        if (checkpoints[s] <= prev) return GRAFT_ERR_INVALID_ARG;
        prev = checkpoints[s];
        if (checkpoints[s] >= D) continue;  // unreachable checkpoint: dropped
        if (ncp == GRAFT_MAX_CHECKPOINTS) return GRAFT_ERR_UNSUPPORTED_SHAPE;
        cfg->checkpoint[ncp] = checkpoints[s];
        cfg->tau[ncp] = tau[s];
        ++ncp;
    }
    cfg->n_checkpoints = ncp;
    const long long full_pool = k + (long long)(D - 1) * k * k;
    if (full_pool < Kmax - 1) return GRAFT_ERR_INVALID_ARG;
    int n_tmpl = 0;
    for (int s = 0; s < ncp; ++s) {
        const long long d = cfg->checkpoint[s];
        const long long pool = k + d * k * k;
        const long long lin = ((long long)(Kmax - 1) * (d + 1)) / D;
        cfg->K_draft[s] = (int32_t)(1 + std::min(pool, lin));
        n_tmpl = std::max(n_tmpl, Kmax - cfg->K_draft[s]);
    }
    cfg->K_draft[ncp] = Kmax;
    cfg->n_tmpl = n_tmpl;
    int rc = graft::build_envelope(D, W, n_tmpl, cfg->tmpl_parent, cfg->tmpl_rank);
    if (rc != GRAFT_OK) return rc;
    return graft_config_validate(cfg);
}

extern "C" int graft_config_no_retrieval(GraftConfig* cfg) {
    if (cfg == nullptr) return GRAFT_ERR_INVALID_ARG;
    const int rc = graft_config_validate(cfg);
    if (rc != GRAFT_OK) return rc;
    for (int s = 0; s <= cfg->n_checkpoints; ++s) cfg->K_draft[s] = cfg->Kmax;
    cfg->n_tmpl = 0;
    return graft_config_validate(cfg);
}

extern "C" const char* graft_status_string(int code) {
    switch (code) {
        case GRAFT_OK: return "ok";
        case GRAFT_ERR_INVALID_ARG: return "invalid argument";
        case GRAFT_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case GRAFT_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
        case GRAFT_ERR_CUDA: return "CUDA launch or device query failed";
        default: return "unknown graft status";
    }
}

extern "C" int graft_version(void) { return 100; }

extern "C" uint64_t graft_launch_count(void) { return graft::g_launches.load(std::memory_order_relaxed); }

extern "C" const char* graft_last_cuda_error(void) { return cudaGetErrorName(graft::g_last_cuda_error); }
