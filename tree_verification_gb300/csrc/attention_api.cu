// graft_tree_attention: argument checks, key-chunk policy and dispatch.
//
// The chunk size is chosen from the cache capacity so that the number of
// CTAs is about the device's SM count (small batches, long prefixes) while
// each chunk stays long enough that partial outputs are a small fraction of
// the KV bytes read.  The same policy sizes the workspace.
#include "attention.cuh"
#include "common.cuh"

namespace graft {
namespace {

struct AttnPlan {
    int G, R, nRB, C, nchunk, tiles;
    int persist;  // > 0: CTAs of the persistent two-tile kernel
    bool stream;  // persistent kernel with the stream schedule
    bool tc;
};

// Key-chunk policy: each (request, KV head, row block) gets as many chunk
// CTAs as keep one CTA per SM busy (no partial second wave), but no more than
// the cache capacity can fill with chunks of at least kMinChunk keys, so the
// partial outputs stay a modest share of the KV bytes.  Each CTA then derives
// its request's chunk length from the request's own key count (chunk_len in
// attention.cuh), so the split does not depend on how far the cache capacity
// exceeds the prefixes.
//
// Row blocks: on the tcgen05 path a CTA takes two 128-row tiles that share
// every K/V block, unless that plan would leave each CTA of a full-capacity
// request fewer than 1024 keys; then one tile per CTA (twice the CTAs, a
// shorter prologue) does better.  A single row block always goes to the
// two-tile kernel.
//
// Persistence: when the two-tile grid would need more than one wave (more
// work items than SMs) and the row tiles pair up (an even tile count), one
// CTA per SM runs the items back to back (attention_tcp.cu), which hides each
// item's start and finish behind its neighbours and deals items of
// decreasing length evenly.  On request (GraftAttnTuning.split = 1), with
// one key chunk per request and at most 256 requests, the stream kernel
// splits the items' key blocks evenly over the CTAs instead, cut items
// merged by their last piece.
//
// The plan depends only on the call's shape, the device's SM count and the
// optional GraftAttnTuning overrides, never on the process environment, so a
// workspace sized for a shape fits every call of that shape.
constexpr long long kMinChunk = 256;

long long chunk_count(long long Lcap, long long units, int sms, long long min_chunk) {
    long long target = sms / units;
    if (target < 1) target = 1;
    const long long fill = Lcap > 0 ? (Lcap + min_chunk - 1) / min_chunk : 1;
    return target < fill ? target : fill;
}

int check_tuning(const GraftAttnTuning* t) {
    if (t == nullptr) return GRAFT_OK;
    if (t->tiles != 0 && t->tiles != 1 && t->tiles != 2) return GRAFT_ERR_INVALID_ARG;
    if (t->min_chunk < 0 || t->persist_ctas < -1 || t->split < 0 || t->split > 1 || t->wait_ns < 0)
        return GRAFT_ERR_INVALID_ARG;
    for (int i = 0; i < 3; ++i)
        if (t->reserved[i] != 0) return GRAFT_ERR_INVALID_ARG;
    return GRAFT_OK;
}

AttnPlan plan_attention(int B, int Hq, int Hkv, int Kmax, int64_t Lcap, const GraftAttnTuning* tune) {
    AttnPlan p;
    p.G = Hq / Hkv;
    p.R = Kmax * p.G;
    p.nRB = (p.R + 127) / 128;
    p.tc = attn_tc_supported(p.G);
    int sms = device_sm_count();
    if (sms <= 0) sms = 148;
    constexpr long long blk = ATTN_TC_BLOCK_KEYS;
    long long min_chunk = kMinChunk;
    if (tune != nullptr && tune->min_chunk > 0) min_chunk = (tune->min_chunk + blk - 1) / blk * blk;
    if (min_chunk > (1LL << 30)) min_chunk = 1LL << 30;
    p.tiles = 1;
    if (p.tc) {
        const long long units2 = (long long)B * Hkv * ((p.nRB + 1) / 2);
        const long long n2 = chunk_count(Lcap, units2, sms, min_chunk);
        // with a single row block both kernels run the same grid; the two-tile kernel is quicker
        p.tiles = (p.nRB == 1 || (Lcap + n2 - 1) / n2 >= 1024) ? 2 : 1;
        if (tune != nullptr && tune->tiles != 0) p.tiles = tune->tiles;
    }
    const long long units = (long long)B * Hkv * ((p.nRB + p.tiles - 1) / p.tiles);
    p.C = (int)min_chunk;
    p.nchunk = (int)chunk_count(Lcap, units, sms, min_chunk);
    p.persist = 0;
    if (p.tc && p.tiles == 2 && p.nRB % 2 == 0) {
        const long long items = (long long)B * p.nchunk * Hkv * (p.nRB / 2);
        const int force = tune != nullptr ? tune->persist_ctas : 0;
        if (force > 0)
            p.persist = (int)(items < force ? items : force);
        else if (force == 0 && items > sms)
            p.persist = sms;
    }
    p.stream = p.persist > 0 && p.nchunk == 1 && B <= 256 && tune != nullptr && tune->split == 1 &&
               (long long)B * Hkv * (Lcap / ATTN_TC_BLOCK_KEYS + 4) < (1LL << 30);  // cost units fit an int
    if (p.stream) {
        // CTAs come in groups of one per row-tile pair of a (request, KV head)
        const int pairs = p.nRB / 2;
        const int want = (tune != nullptr && tune->persist_ctas > 0) ? tune->persist_ctas : sms;
        p.persist = (want / pairs > 0 ? want / pairs : 1) * pairs;
    }
    return p;
}

// Workspace: the stream schedule's arrival counters come first (the part the caller zeroes once and
// every call leaves at zero), then the partial rows.
size_t attn_ws(const AttnPlan& p, int B, int Hkv, AttnArgs* a, void* ws) {
    WsCarver c(ws);
    const size_t items = p.stream ? (size_t)B * Hkv * (p.nRB / 2) : 0;
    int32_t* cnt = c.take<int32_t>(items * 2);
    const size_t cut_rows = p.stream ? (size_t)2 * p.persist * 2 * 128 : 0;
    float* co = c.take<float>(cut_rows * GRAFT_HEAD_DIM);
    float* cl = c.take<float>(cut_rows);
    const size_t parts = p.nchunk > 1 ? (size_t)B * Hkv * p.nRB * p.nchunk * 128 : 0;
    float* po = c.take<float>(parts * GRAFT_HEAD_DIM);
    float* pl = c.take<float>(parts);
    if (a) {
        a->part_o = po;
        a->part_lse = pl;
        a->cut_cnt = cnt;
        a->cut_o = co;
        a->cut_lse = cl;
    }
    return c.bytes();
}

int check_shape(int B, int Hq, int Hkv, int head_dim, int Kmax, int64_t Lcap) {
    if (B < 0 || Hq < 1 || Hkv < 1 || Kmax < 1 || Lcap < 0) return GRAFT_ERR_INVALID_ARG;
    if (head_dim != GRAFT_HEAD_DIM) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    if (Hq % Hkv != 0) return GRAFT_ERR_INVALID_ARG;
    if (Kmax > GRAFT_MAX_KMAX) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    if ((long long)Kmax * (Hq / Hkv) > 1024) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    if (Lcap > (1LL << 30)) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    if (B > 65535) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    return GRAFT_OK;
}

}  // namespace
}  // namespace graft

using namespace graft;

extern "C" int graft_tree_attention_workspace_size_ex(int B, int Hq, int Hkv, int head_dim, int Kmax, int64_t Lcap,
                                                      const GraftAttnTuning* tuning, size_t* bytes) {
    if (bytes == nullptr) return GRAFT_ERR_INVALID_ARG;
    int rc = check_shape(B, Hq, Hkv, head_dim, Kmax, Lcap);
    if (rc == GRAFT_OK) rc = check_tuning(tuning);
    if (rc != GRAFT_OK) return rc;
    const AttnPlan p = plan_attention(B, Hq, Hkv, Kmax, Lcap, tuning);
    *bytes = attn_ws(p, B, Hkv, nullptr, nullptr);
    return GRAFT_OK;
}

extern "C" int graft_tree_attention_workspace_size(int B, int Hq, int Hkv, int head_dim, int Kmax, int64_t Lcap,
                                                   size_t* bytes) {
    return graft_tree_attention_workspace_size_ex(B, Hq, Hkv, head_dim, Kmax, Lcap, nullptr, bytes);
}

extern "C" int graft_tree_attention_ex(int B, int Hq, int Hkv, int head_dim, int Kmax, const void* Q, const void* Kc,
                                       const void* Vc, int64_t Lcap, const void* Kt, const void* Vt, const int32_t* L,
                                       const uint64_t* tree_mask, float scale, void* O, int32_t* status,
                                       const GraftAttnTuning* tuning, void* ws, size_t ws_bytes,
                                       graft_stream_t stream) {
    int rc = check_shape(B, Hq, Hkv, head_dim, Kmax, Lcap);
    if (rc == GRAFT_OK) rc = check_tuning(tuning);
    if (rc != GRAFT_OK) return rc;
    if (B == 0) return GRAFT_OK;
    if (Q == nullptr || Kt == nullptr || Vt == nullptr || L == nullptr || tree_mask == nullptr || O == nullptr)
        return GRAFT_ERR_INVALID_ARG;
    if (Lcap > 0 && (Kc == nullptr || Vc == nullptr)) return GRAFT_ERR_INVALID_ARG;
    const uintptr_t al = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(Kc) |
                         reinterpret_cast<uintptr_t>(Vc) | reinterpret_cast<uintptr_t>(Kt) |
                         reinterpret_cast<uintptr_t>(Vt) | reinterpret_cast<uintptr_t>(O);
    if (al & 15) return GRAFT_ERR_INVALID_ARG;  // 16-byte vector loads and stores
    const AttnPlan p = plan_attention(B, Hq, Hkv, Kmax, Lcap, tuning);
    const size_t need = attn_ws(p, B, Hkv, nullptr, nullptr);
    if (!ws_ok(ws, ws_bytes, need)) return GRAFT_ERR_WORKSPACE;
    AttnArgs a{};
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = p.G;
    a.Kmax = Kmax;
    a.R = p.R;
    a.nRB = p.nRB;
    a.tiles = p.tiles;
    a.C = p.C;
    a.nchunk = p.nchunk;
    a.Lcap = (int)Lcap;
    a.scale = scale;
    a.wait_ns = (tuning != nullptr && tuning->wait_ns > 0) ? (uint64_t)tuning->wait_ns : 500000000ull;
    a.Q = Q;
    a.Kc = Kc;
    a.Vc = Vc;
    a.Kt = Kt;
    a.Vt = Vt;
    a.L = L;
    a.mask = tree_mask;
    a.O = O;
    a.status = status;
    attn_ws(p, B, Hkv, &a, ws);
    if ((long long)p.nRB * Hkv > 65535LL || p.nchunk > 65535) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    // the persistent kernels store output rows in 32-byte pieces
    if (p.persist > 0 && (reinterpret_cast<uintptr_t>(O) & 31) == 0)
        return p.stream ? attn_tcs_launch(a, p.persist, (cudaStream_t)stream)
                        : attn_tcp_launch(a, p.persist, (cudaStream_t)stream);
    // (an O only 16-byte aligned runs the two-tile kernel, which needs no workspace with one chunk)
    if (p.tc) return p.tiles == 2 ? attn_tc_launch(a, (cudaStream_t)stream) : attn_tc1_launch(a, (cudaStream_t)stream);
    return attn_mma_launch(a, (cudaStream_t)stream);
}

extern "C" int graft_tree_attention(int B, int Hq, int Hkv, int head_dim, int Kmax, const void* Q, const void* Kc,
                                    const void* Vc, int64_t Lcap, const void* Kt, const void* Vt, const int32_t* L,
                                    const uint64_t* tree_mask, float scale, void* O, int32_t* status, void* ws,
                                    size_t ws_bytes, graft_stream_t stream) {
    return graft_tree_attention_ex(B, Hq, Hkv, head_dim, Kmax, Q, Kc, Vc, Lcap, Kt, Vt, L, tree_mask, scale, O,
                                   status, nullptr, ws, ws_bytes, stream);
}
