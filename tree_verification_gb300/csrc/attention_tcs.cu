// Tree-masked GQA attention on the 5th-generation tensor cores, persistent
// two-tile kernel with the key blocks split evenly over its CTAs ("stream"
// schedule), for grids of several waves with one key chunk per request.
//
// Graft article, architecture paragraph: the hybrid tree is verified on the
// standard tree-attention path in one target forward; Graft abstract: large
// draft trees cost VRAM bandwidth and compute.  Each query row (tree node i,
// query head h) attends to its request's L prefix keys and to the tree keys
// in node i's ancestor-or-self mask, with KV head h / group.
//
// A work item is two 128-row tiles of one (request, KV head) against all of
// the request's keys (the prefix in 128-key blocks, then the tree block),
// items ordered longest request first.  The work of every (request, KV head)
// forms one sequence in cost units: ITEM_COST units that stand for an item's
// fixed cost (Q load, the last product's latency, the epilogue: about two
// blocks' time), then its blocks.  The CTAs form groups of one CTA per
// row-tile pair; group p of P takes the units [p S, (p + 1) S), S =
// ceil(total / P), and each of its CTAs runs its own row-tile pair over the
// blocks in that range, so the pairs that read the same K/V run in step (one
// HBM read, L2 hits for the others) and every SM gets the same work to
// within one block.  An item whose blocks straddle a group boundary runs in
// pieces by consecutive groups (a boundary inside an item's fixed-cost units
// hands the whole item to the next group).  Each piece writes its rows as a
// normalised float32 partial with its log2-sum-exp to a slot of its CTA,
// fences, and adds one to the item's arrival counter; the piece that arrives
// last merges every piece's partial into the bf16 output and resets the
// counter to zero.  No CTA waits for another.  The counters live in the
// workspace, which the caller zeroes once; every completed call leaves them
// at zero.
//
// The pipeline is the persistent kernel's (attention_tcp.cu): K and V rings
// running across pieces with running stage and phase counters, the next
// piece's Q tiles loaded once the current piece's last S product has run,
// the epilogue writing rows from registers after signalling that the next
// piece's first PV may overwrite O in TMEM, a single-thread MMA issuer that
// tests the next group's barrier before the last two products of the
// current group, and free-running exponentials of the two tiles; TMEM
// layout, masking and lazy rescale are the two-tile kernel's.
//
// Every mbarrier wait is bounded; on timeout the CTA raises
// GRAFT_STATUS_TIMEOUT, stops issuing work, drains what it issued (again
// with a bound) and frees its TMEM before returning.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>

#include "attention.cuh"
#include "common.cuh"
#include "tc_ptx.cuh"

namespace graft {
namespace attn_tcs {

using namespace tc;

constexpr int HD = GRAFT_HEAD_DIM;
constexpr int BN = ATTN_TC_BLOCK_KEYS;  // keys per block
constexpr int SK = 2;                   // K ring depth
constexpr int SV = 3;                   // V ring depth
constexpr int NTHREADS = 320;
constexpr int MAX_ORDER = 256;          // requests ranked by length in shared memory (ids fit a byte)
constexpr int ITEM_COST = 2;            // stream schedule: an item's fixed cost, in 128-key blocks
constexpr uint32_t BOX_BYTES = BN * 64 * 2;             // one box: 128 keys (or rows) x 64 dims bf16
constexpr uint32_t BLK_BYTES = 2 * BOX_BYTES;           // one K or V block (128 keys x 128 dims)
constexpr uint32_t Q_TILE_BYTES = 2 * 128 * 64 * 2;     // 128 rows x 128 dims
// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + 2 * Q_TILE_BYTES;
constexpr uint32_t OFF_V = OFF_K + SK * BLK_BYTES;
constexpr uint32_t OFF_BAR = OFF_V + SV * BLK_BYTES;
// barriers
constexpr int BAR_Q = 0;              // an item's Q tiles landed (one phase per item)
constexpr int BAR_KF = 1;             // [SK] K block landed
constexpr int BAR_KE = BAR_KF + SK;   // [SK] K block consumed by both S products
constexpr int BAR_VF = BAR_KE + SK;   // [SV] V block landed
constexpr int BAR_VE = BAR_VF + SV;   // [SV] V block consumed by both PV products
constexpr int BAR_S = BAR_VE + SV;    // [tile] S_t ready in TMEM
constexpr int BAR_P = BAR_S + 2;      // [tile] P_t written to TMEM (128 arrivals)
constexpr int BAR_DONE = BAR_P + 2;   // an item's MMAs completed (one phase per item)
constexpr int BAR_OFREE = BAR_DONE + 1;  // [tile] an item's O_t read out of TMEM (128 arrivals)
// a CTA runs at most two cut pieces, its first (slot kind 0) and its last (kind 1): one-shot barriers
constexpr int BAR_CUT = BAR_OFREE + 2;    // [kind][tile] a cut piece's partial rows written (128 arrivals)
constexpr int BAR_CUTL = BAR_CUT + 4;    // [kind][tile] its arrival counter read (one arrival)
constexpr int N_BARS = BAR_CUTL + 4;
constexpr uint32_t OFF_MISC = OFF_BAR + N_BARS * 8;  // tmem slot, abort flag
constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

constexpr uint32_t TM_S = 0;    // + tile * 128
constexpr uint32_t TM_O = 256;  // + tile * 128
constexpr float RESCALE_LOG2 = 8.f;
// Pipeline waits are bounded by kWaitNs (a.wait_ns in the failure-path tests); the waits of the
// teardown keep fixed bounds, so every issued load and MMA completes before the CTA frees TMEM and exits.
constexpr uint64_t kWaitNs = 500000000ull;      // bound on any pipeline wait (the kernel runs for microseconds)
constexpr uint64_t kTeardownNs = 500000000ull;  // bound on the last MMA completion before TMEM is freed
constexpr uint64_t kDrainNs = 100000000ull;  // bound on draining in-flight loads after an abort

struct Maps {
    CUtensorMap q, kc, vc, kt, vt;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ bool aborted(const volatile uint32_t* flag) { return *flag != 0; }

__device__ __forceinline__ void raise_abort(volatile uint32_t* flag, int32_t* status) {
    *flag = 1;
    flag_status(status, GRAFT_STATUS_TIMEOUT);
}

// 32-byte store (eight 32-bit words) to a 32-byte aligned global address: a warp's 32 rows fill
// whole 32-byte sectors per instruction
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// 16-byte store to p + OFF bytes (16-byte aligned), the offset folded into the instruction so that
// strided stores share one address register
template <int OFF>
__device__ __forceinline__ void st_global_v4(void* p, float x, float y, float z, float w) {
    asm volatile("st.global.v4.f32 [%0+%5], {%1, %2, %3, %4};" ::"l"(p), "f"(x), "f"(y), "f"(z), "f"(w), "n"(OFF)
                 : "memory");
}

// One piece: blocks [jb, je) of the item of (request b, KV head kvh, row-tile pair rb), whose
// blocks are the prefix's (nb_prefix of them, the last one ragged when ragged_valid != 0) and then the
// tree block.
struct Item {
    int b, kvh, rb;
    int nb_prefix, nb, ragged_block, ragged_valid;
    int jb, je;
    int idx;      // the item's arrival counter
    int g_start;  // its first block's cost unit
};

// This CTA's schedule tables in shared memory (file scope, so the walk functions name them without
// holding pointers in registers): requests ranked by length, longest first; in the stream schedule
// the first block of every ranked request (counting each KV head's blocks once), and the blocks per
// CTA group and in all.
__shared__ uint8_t s_order[MAX_ORDER];
__shared__ int s_pref[MAX_ORDER + 1];
__shared__ int s_S, s_T;

__device__ __forceinline__ bool ranked(const AttnArgs& a) { return a.B > 1; }  // the launch keeps B <= MAX_ORDER
__device__ __forceinline__ int ranked_request(const AttnArgs& a, int z) { return ranked(a) ? s_order[z] : z; }

// A position in this CTA's walk: the next cost unit of the sequence.
__device__ __forceinline__ int walk_start(const AttnArgs& a) { return min((int)blockIdx.x / (a.nRB / 2) * s_S, s_T); }

// The arguments the walk reads, passed by value to its out-of-line search.
struct WalkArgs {
    int B, Hkv, nRB;
    const int32_t* L;
};

// The next piece of this CTA's walk; false past the end of its group's range.
__device__ __forceinline__ bool next_item_search(int& w, const WalkArgs& a, Item& it) {
    const int nrb2 = a.nRB / 2;
    const int S = s_S;
    const int g_end = min(((int)blockIdx.x / nrb2 + 1) * S, s_T);
    if (w >= g_end) return false;
    // the request whose blocks hold w: the last z with pref[z] <= w (its block count is not zero)
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_pref[mid] <= w) lo = mid;
        else hi = mid - 1;
    }
    const int z = lo;
    const int cz = (s_pref[z + 1] - s_pref[z]) / a.Hkv;  // an item's cost: ITEM_COST + its blocks
    const int local = w - s_pref[z];
    const int kvh = local / cz;
    const int c0 = s_pref[z] + kvh * cz;                 // the item's first cost unit
    const int b0 = c0 + ITEM_COST;                       // its first block's cost unit
    if (g_end <= b0) {
        // the range ends inside the item's fixed-cost units: the next group runs the whole item
        w = g_end;
        return false;
    }
    const int b = a.B > 1 ? s_order[z] : z;  // requests ranked by length (the launch keeps B <= MAX_ORDER)
    const int Lb = a.L[b];  // in [0, Lcap]: requests outside it hold no blocks
    it.b = b;
    it.kvh = kvh;
    it.rb = (int)blockIdx.x % nrb2;  // this CTA's row-tile pair in its group
    it.nb_prefix = (Lb + BN - 1) / BN;
    it.nb = it.nb_prefix + 1;
    it.ragged_valid = Lb % BN;
    it.ragged_block = it.ragged_valid != 0 ? it.nb_prefix - 1 : -1;
    it.idx = (z * a.Hkv + kvh) * nrb2 + it.rb;
    it.g_start = b0;
    it.jb = max(w, b0) - b0;
    it.je = min(cz - ITEM_COST, g_end - b0);
    w = b0 + it.je;  // the item's end (its last cost unit + 1) when its last block is in the range
    return true;
}

struct NextItem {
    Item it;
    int w;
    bool live;
};

// The search runs once per piece; kept out of line (and out of the block loops that call it), it
// leaves those loops small in the instruction cache.
__device__ __noinline__ NextItem next_item_ool(int w, WalkArgs wa) {
    NextItem r;
    r.w = w;
    r.live = next_item_search(r.w, wa, r.it);
    return r;
}

__device__ __forceinline__ bool next_item(int& w, const AttnArgs& a, Item& it) {
    const NextItem r = next_item_ool(w, WalkArgs{a.B, a.Hkv, a.nRB, a.L});
    w = r.w;
    it = r.it;
    return r.live;
}

// A position (item, block) in this CTA's stream of blocks, with the few item fields the TMA
// producer reads (it holds four of these).
struct Cursor {
    int w;
    bool live;
    int b, kvh, rb, nb_prefix, jb, je;
    int j;  // block of the item, in [jb, je)
};

__device__ __forceinline__ void cursor_next(Cursor& cu, const AttnArgs& a) {
    Item it;
    cu.live = next_item(cu.w, a, it);
    cu.b = it.b;
    cu.kvh = it.kvh;
    cu.rb = it.rb;
    cu.nb_prefix = it.nb_prefix;
    cu.jb = it.jb;
    cu.je = it.je;
    cu.j = cu.live ? it.jb : 0;
}

__device__ __forceinline__ void cursor_start(Cursor& cu, const AttnArgs& a) {
    cu.w = walk_start(a);
    cursor_next(cu, a);
}

__device__ __forceinline__ void advance(Cursor& cu, const AttnArgs& a) {
    if (!cu.live) return;
    if (++cu.j < cu.je) return;
    cursor_next(cu, a);
}

// Stream schedule: the partial slot of the piece of an item that CTA q runs.  A CTA's cut pieces can
// only sit at the two ends of its group's range: a piece that starts inside its item (jb > 0, the
// item began in an earlier group) opens the range and takes slot 2q; the item's first piece (cut at
// the range's end) closes it and takes slot 2q + 1.
__device__ __forceinline__ int cut_slot(bool first_piece, int q) { return first_piece ? 2 * q + 1 : 2 * q; }

// kTestWaits: pipeline waits bounded by a.wait_ns (the failure-path tests); otherwise by kWaitNs, a
// compile-time constant, so the production instantiation carries no run-time bound.
// The last arriving piece of a cut item merges every piece's normalised fp32 partial into the bf16
// output row of thread r (one row per thread, tile t): weights 2^(lse_i - max), loads issued in batches
// before they are used (every piece's log2-sum-exp, then two pieces' 16 columns at a time).  Out of
// line: it runs once per cut item, and keeping it out of the kernel body keeps the hot loops' code
// compact (a larger kernel body measured slower per key block).
__device__ __noinline__ void merge_cut_pieces(const float* __restrict__ cut_lse, const float* __restrict__ cut_o,
                                              __nv_bfloat16* orow, int q_first, int np, int nrb2, int rb, int t,
                                              int r) {
    // slot-tile index of piece i (its log2-sum-exp row is (index) * 128 + r)
    auto row_of = [&](int i) -> size_t {
        const int qq = q_first + i;
        return (size_t)cut_slot(qq == q_first, qq * nrb2 + rb) * 2 + t;
    };
    float mx = -INFINITY;
    for (int i0 = 0; i0 < np; i0 += 4) {
        float l4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) l4[u] = i0 + u < np ? __ldcg(cut_lse + row_of(i0 + u) * 128 + r) : -INFINITY;
#pragma unroll
        for (int u = 0; u < 4; ++u) mx = fmaxf(mx, l4[u]);
    }
    float wsum = 0.f;
    for (int i0 = 0; i0 < np; i0 += 4) {
        float l4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) l4[u] = i0 + u < np ? __ldcg(cut_lse + row_of(i0 + u) * 128 + r) : -INFINITY;
#pragma unroll
        for (int u = 0; u < 4; ++u) wsum += i0 + u < np ? ex2(l4[u] - mx) : 0.f;
    }
    const float winv = wsum > 0.f ? 1.f / wsum : 0.f;
    for (int c0 = 0; c0 < HD; c0 += 16) {
        float4 acc[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) acc[x] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i0 = 0; i0 < np; i0 += 2) {
            float4 v[2][4];
            float wq[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const bool live = i0 + u < np;
                const size_t st = live ? row_of(i0 + u) : 0;
                wq[u] = live ? ex2(__ldcg(cut_lse + st * 128 + r) - mx) : 0.f;
                const float4* src = reinterpret_cast<const float4*>(cut_o) + (st * (HD / 4) + c0 / 4) * 128 + r;
#pragma unroll
                for (int x = 0; x < 4; ++x) v[u][x] = live ? __ldcg(src + x * 128) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    acc[x].x += wq[u] * v[u][x].x;
                    acc[x].y += wq[u] * v[u][x].y;
                    acc[x].z += wq[u] * v[u][x].z;
                    acc[x].w += wq[u] * v[u][x].w;
                }
        }
        uint32_t wd[8];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc[y].x * winv, acc[y].y * winv);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc[y].z * winv, acc[y].w * winv);
            wd[2 * y] = *reinterpret_cast<uint32_t*>(&lo);
            wd[2 * y + 1] = *reinterpret_cast<uint32_t*>(&hi);
        }
        st_global_v8(orow + c0, wd);
    }
}

template <bool kTestWaits>
__global__ void __launch_bounds__(NTHREADS, 1)
attn_tcs_kernel(const __grid_constant__ Maps maps, AttnArgs a) {
    const uint64_t wait_ns = kTestWaits ? a.wait_ns : kWaitNs;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_last[2];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + OFF_MISC);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + OFF_MISC + 4);
    auto bar = [&](int i) { return base + OFF_BAR + 8u * (uint32_t)i; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nrb2 = a.nRB / 2;  // row-tile pairs per (request, KV head); the launch needs nRB even

    // Prologue that touches no global memory: it overlaps the previous kernel's tail.
    if (tid == 0) {
        for (int i = 0; i < N_BARS; ++i) {
            uint32_t cnt = 1;
            if (i == BAR_P || i == BAR_P + 1 || i == BAR_OFREE || i == BAR_OFREE + 1 ||
                (i >= BAR_CUT && i < BAR_CUT + 4))
                cnt = 128;
            mbar_init(bar(i), cnt);
        }
        *abort_flag = 0;
        fence_mbar_init();
    } else if (tid == 32) {
        tma_prefetch_desc(&maps.vc);
        tma_prefetch_desc(&maps.vt);
    } else if (tid == 64) {
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.kc);
        tma_prefetch_desc(&maps.kt);
    }
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(base + OFF_MISC, 512);
        tmem_relinquish();
        tc_fence_before();
    }
    griddep_wait();
    griddep_launch_dependents();
    // rank of every request's length, longest first (ties to the lower index)
    if (ranked(a) && tid < a.B) {
        const int li = a.L[tid];
        int rank = 0;
        for (int j = 0; j < a.B; ++j) {
            const int lj = a.L[j];
            rank += (lj > li) || (lj == li && j < tid);
        }
        s_order[rank] = (uint8_t)tid;
    }
    {
        // cost of every ranked request (all its items), then the running sum; the launch keeps
        // B <= MAX_ORDER and one key chunk per request
        __syncthreads();
        if (tid < a.B) {
            const int b = ranked_request(a, tid);
            const int Lb = a.L[b];
            const bool bad = Lb < 0 || Lb > a.Lcap;
            if (bad && blockIdx.x == 0) flag_status(a.status, GRAFT_STATUS_LENGTH);
            s_pref[tid + 1] = bad ? 0 : ((Lb + BN - 1) / BN + 1 + ITEM_COST) * a.Hkv;
        }
        __syncthreads();
        if (warp == 0) {
            // inclusive scan of s_pref[1..B] by one warp: eight entries per lane, then across lanes
            const int per = (a.B + 31) / 32;
            int run = 0;
            for (int x = 0; x < per; ++x) {
                const int z = lane * per + x;
                if (z < a.B) run += s_pref[z + 1];
            }
            int incl = run;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            int acc = incl - run;
            for (int x = 0; x < per; ++x) {
                const int z = lane * per + x;
                if (z < a.B) {
                    acc += s_pref[z + 1];
                    s_pref[z + 1] = acc;
                }
            }
            __syncwarp();  // every lane's running sums are written before lane 0 reads the total
            if (lane == 0) {
                s_pref[0] = 0;
                s_T = s_pref[a.B];
                const int groups = (int)gridDim.x / nrb2;  // the launch makes gridDim.x a multiple of nrb2
                s_S = (s_T + groups - 1) / groups;
            }
        }
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    int k_issued = 0, v_issued = 0, q_issued = 0;  // blocks and Q pairs the producer has armed
    int ndone = 0;                   // DONE commits of the MMA issuer
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (lane 0)
        if (lane == 0) {
            auto load_q = [&](const Cursor& cu) {
                ++q_issued;
                mbar_expect_tx(bar(BAR_Q), 2 * Q_TILE_BYTES);
                for (int t = 0; t < 2; ++t) {
                    const int nz = cu.b * a.Kmax + (cu.rb * 256 + t * 128) / a.G;
                    for (int h = 0; h < 2; ++h)
                        tma_load_3d(base + OFF_Q + t * Q_TILE_BYTES + h * (Q_TILE_BYTES / 2), &maps.q, bar(BAR_Q),
                                    h * 64, cu.kvh * a.G, nz);
                }
            };
            auto load_block = [&](const Cursor& cu, const CUtensorMap* prefix_map, const CUtensorMap* tree_map,
                                  uint32_t dst, uint32_t full) {
                mbar_expect_tx(full, BLK_BYTES);
                for (int h = 0; h < 2; ++h) {
                    if (cu.j < cu.nb_prefix)
                        tma_load_4d(dst + h * BOX_BYTES, prefix_map, full, h * 64, cu.kvh, cu.j * BN, cu.b);
                    else
                        tma_load_4d(dst + h * BOX_BYTES, tree_map, full, h * 64, cu.kvh, 0, cu.b);
                }
            };
            auto load_k = [&](Cursor& cu) {
                load_block(cu, &maps.kc, &maps.kt, base + OFF_K + (k_issued % SK) * BLK_BYTES,
                           bar(BAR_KF + k_issued % SK));
                ++k_issued;
                advance(cu, a);
            };
            auto load_v = [&](Cursor& cu) {
                load_block(cu, &maps.vc, &maps.vt, base + OFF_V + (v_issued % SV) * BLK_BYTES,
                           bar(BAR_VF + v_issued % SV));
                ++v_issued;
                advance(cu, a);
            };
            Cursor kc;
            cursor_start(kc, a);
            Cursor vc = kc, cc = kc;
            if (kc.live) load_q(kc);
            for (int s = 0; s < SK && kc.live; ++s) load_k(kc);
            for (int s = 0; s < SV && vc.live; ++s) load_v(vc);
            // Stages are released in the tensor pipe's order S_1(g), PV_1(g), S_1(g + 1), ..., so
            // one thread that waits for each release in turn never waits behind a later one.
            for (int g = 0; cc.live; ++g) {
                Cursor nx = cc;
                advance(nx, a);
                const bool next_q = nx.live && nx.j == nx.jb;  // block g ends its piece: the next Q follows
                if (kc.live || next_q) {
                    if (!mbar_wait(bar(BAR_KE + g % SK), (g / SK) & 1, wait_ns)) {
                        raise_abort(abort_flag, a.status);
                        break;
                    }
                    if (aborted(abort_flag)) break;
                    // every S product of the piece has run: its Q tiles are free
                    if (next_q) load_q(nx);
                    if (kc.live) load_k(kc);
                }
                if (vc.live) {
                    if (!mbar_wait(bar(BAR_VE + g % SV), (g / SV) & 1, wait_ns)) {
                        raise_abort(abort_flag, a.status);
                        break;
                    }
                    if (aborted(abort_flag)) break;
                    load_v(vc);
                }
                cc = nx;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (lane 0 alone)
        // tcgen05.mma issue hardly queues ahead of the tensor pipe, so every cycle this thread
        // spends between two products, waits included, is a cycle the pipe idles: one thread runs
        // the loop with running ring counters, and the barrier the next group of products needs is
        // tested (non-blocking) just before the last two products of the current group.
        if (lane == 0) {
            const uint32_t idS = idesc_bf16(128, BN, false, false);
            const uint32_t idO = idesc_bf16(128, HD, false, true);
            // Descriptors are built once; each MMA adds a byte offset (in 16-byte units) to the
            // start-address field, which sits in the low bits and cannot carry out of them here
            // (every shared-memory address is below 256 KB).
            const uint64_t q_desc = sdesc_sw128(base + OFF_Q, 16, 1024);
            const uint64_t k_desc = sdesc_sw128(base + OFF_K, 16, 1024);
            const uint64_t v_desc = sdesc_sw128(base + OFF_V, BOX_BYTES, 1024);
            int kst = 0, kph = 0;  // K ring: stage and phase of the next block the S products read
            int vst = 0, vph = 0;  // V ring: stage and phase of the next block the PV products read
            uint32_t pph = 0;      // phase of the S and P barriers of the current block (g & 1)
            // (plain values, no references: address-taken locals would live in local memory)
            struct Pre {
                int bar;  // barrier index, -1: none
                uint32_t ph;
            };
            const Pre none{-1, 0u};
            auto test_pre = [&](Pre pre) -> bool { return pre.bar < 0 || mbar_test_now(bar(pre.bar), pre.ph); };
            auto wait_pre = [&](Pre pre, bool ready) -> bool {
                return ready || mbar_wait(bar(pre.bar), pre.ph, wait_ns);
            };
            auto group_S = [&](int t, Pre nxt) -> bool {
                bool ready = false;
                const uint64_t kd = k_desc + ((kst * BLK_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    if (kk == HD / 16 - 2) ready = test_pre(nxt);
                    const uint32_t off = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
                    const uint32_t qoff = t * Q_TILE_BYTES + (kk >> 2) * (Q_TILE_BYTES / 2) + (kk & 3) * 32;
                    mma_bf16_ss(tmem + TM_S + t * 128, q_desc + (qoff >> 4), kd + (off >> 4), idS, kk > 0);
                }
                mma_commit(bar(BAR_S + t));
                if (t == 1) {
                    mma_commit(bar(BAR_KE + kst));
                    if (++kst == SK) { kst = 0; kph ^= 1; }
                }
                return ready;
            };
            auto group_PV = [&](int t, bool first, Pre nxt) -> bool {
                bool ready = false;
                const uint64_t vd = v_desc + ((vst * BLK_BYTES) >> 4);
                const uint32_t p = tmem + TM_S + t * 128;  // P_t as packed bf16 pairs
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    if (kk == BN / 16 - 2) ready = test_pre(nxt);
                    mma_bf16_ts(tmem + TM_O + t * 128, p + kk * 8, vd + ((kk * 2048) >> 4), idO, !first || kk > 0);
                }
                if (t == 1) mma_commit(bar(BAR_VE + vst));
                return ready;
            };
            bool ok = true;
            int q = 0;  // pieces issued
            int w = walk_start(a);
            Item it;
            while (ok && next_item(w, a, it)) {
                ok = mbar_wait(bar(BAR_Q), q & 1, wait_ns) && !aborted(abort_flag) &&
                     mbar_wait(bar(BAR_KF + kst), kph, wait_ns);
                if (!ok) break;
                tc_fence_after();
                group_S(0, none);
                Pre vf{BAR_VF + vst, (uint32_t)vph};
                bool vf_ready = group_S(1, vf);
                for (int j = it.jb; j < it.je && ok; ++j) {
                    // (tile 0's softmax warps zero a ragged block's V rows past the chunk end before
                    // they signal P_0, so PV_0 and PV_1, issued after that signal, read zeros there)
                    const bool more = j + 1 < it.je;
                    const bool first = j == it.jb;
                    ok = wait_pre(vf, vf_ready) && mbar_wait(bar(BAR_P), pph, wait_ns);
                    // the piece's first PV overwrites O_t: the previous piece's epilogue must have read it
                    if (ok && first && q > 0) ok = mbar_wait(bar(BAR_OFREE), (q - 1) & 1, wait_ns);
                    if (!ok) break;
                    tc_fence_after();
                    const Pre kf{BAR_KF + kst, (uint32_t)kph};
                    const Pre p1{BAR_P + 1, pph};
                    bool p1_ready;
                    if (more) {
                        const bool kf_ready = group_PV(0, first, kf);
                        // this tile's next S right behind its PV: the other tile's softmax overlaps both
                        ok = wait_pre(kf, kf_ready);
                        if (!ok) break;
                        tc_fence_after();
                        p1_ready = group_S(0, p1);
                    } else {
                        p1_ready = group_PV(0, first, p1);
                    }
                    ok = wait_pre(p1, p1_ready);
                    if (ok && first && q > 0) ok = mbar_wait(bar(BAR_OFREE + 1), (q - 1) & 1, wait_ns);
                    if (!ok) break;
                    tc_fence_after();
                    const int vst_next = vst + 1 == SV ? 0 : vst + 1;
                    const int vph_next = vst + 1 == SV ? vph ^ 1 : vph;
                    vf = Pre{BAR_VF + vst_next, (uint32_t)vph_next};
                    group_PV(1, first, none);
                    vf_ready = more ? group_S(1, vf) : false;
                    vst = vst_next;
                    vph = vph_next;
                    pph ^= 1u;
                }
                // the piece's MMAs (and everything before them) complete: its epilogue may read O
                mma_commit(bar(BAR_DONE));
                ++ndone;
                ++q;
            }
            if (!ok && !aborted(abort_flag)) raise_abort(abort_flag, a.status);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int t = (warp - 2) >> 2;
        const int quad = warp & 3;
        const int r = quad * 32 + lane;  // row within the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const uint32_t sbuf = tmem + lane_base + TM_S + t * 128;
        const float sl2 = a.scale * 1.4426950408889634f;
        bool ok = true;
        int q = 0, g0 = 0;
        int w = walk_start(a);
        while (ok) {
            // The block loop needs only the piece's block range and masks; the item is decoded again
            // for the epilogue (from the walk position), so its fields hold no registers across the loop.
            const int w_item = w;
            int nj, nb_prefix, ragged_block, ragged_valid;  // block counts relative to the piece's first
            uint64_t anc;
            {
                Item it;
                if (!next_item(w, a, it)) break;
                const int gr = (it.rb * 2 + t) * 128 + r;
                anc = gr < a.R ? a.mask[(size_t)it.b * a.Kmax + gr / a.G] : 0ull;
                nj = it.je - it.jb;
                nb_prefix = it.nb_prefix - it.jb;
                ragged_block = it.ragged_block - it.jb;
                ragged_valid = it.ragged_valid;
            }
            float m_used = -INFINITY, l_sum = 0.f;  // running max (log2 units) and row sum
            for (int j = 0; j < nj; ++j) {
                const int g = g0 + j;
                ok = __all_sync(0xffffffffu, mbar_wait(bar(BAR_S + t), g & 1, wait_ns) && !aborted(abort_flag));
                if (!ok) break;
                tc_fence_after();
                if (t == 0 && j == ragged_block) {
                    // zero the V rows past the chunk end (both 64-dim boxes) before PV reads them: the
                    // block's keys there are masked, but the cache rows may hold non-finite garbage
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(BAR_VF + g % SV), (g / SV) & 1, wait_ns));
                    if (!ok) break;
                    uint8_t* v0 = gbase + OFF_V + (g % SV) * BLK_BYTES;
                    for (int x = r; x < (BN - ragged_valid) * 16; x += 128) {
                        const int rr = ragged_valid + x / 16, c16 = x % 16;
                        *reinterpret_cast<uint4*>(v0 + (c16 >= 8 ? BOX_BYTES : 0) + rr * 128 + (c16 & 7) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                const bool tree_blk = j >= nb_prefix;
                float alpha = 1.f;
                bool rescale = false;
                float2 acc;
                float packed[BN / 2];
                // A piece's first block takes its maximum; a later block is first weighed against the
                // running maximum alone and stands if its row sum stays within 2^16 (so no weight
                // passed 2^16: none overflowed, and bf16 P, the fp32 sums and O carry them).  Otherwise
                // it is weighed again with its own maximum; S_t is still intact in TMEM, since P is
                // stored over it only once the block stands.
                for (int pass = 0; pass < 2; ++pass) {
                    float s[BN];
#pragma unroll
                    for (int x = 0; x < BN / 32; ++x) tmem_ld32(sbuf + x * 32, s + x * 32);
                    tmem_wait_ld();
                    if (tree_blk || j == ragged_block) {
                        // only the ragged tail and the tree block need masking: keep-bits for the
                        // block's keys as four 32-bit words (tree keys are < 64, in the ancestor mask)
                        const int valid = tree_blk ? a.Kmax : ragged_valid;
                        uint32_t wd[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const int n = valid - 32 * x;
                            wd[x] = n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
                        }
                        if (tree_blk) {
                            wd[0] &= (uint32_t)anc;
                            wd[1] &= (uint32_t)(anc >> 32);
                            wd[2] = wd[3] = 0u;
                        }
#pragma unroll
                        for (int x = 0; x < BN; ++x) s[x] = ((wd[x >> 5] >> (x & 31)) & 1u) ? s[x] : -INFINITY;
                    }
                    const bool full = j == 0 || pass == 1;
                    if (full) {
                        // block maximum by a tree of pairwise maxima (short dependency chains)
                        float m8[8];
#pragma unroll
                        for (int x = 0; x < 8; ++x) {
                            float m = fmaxf(s[x], s[x + 8]);
#pragma unroll
                            for (int y = 16; y < BN; y += 16) m = fmaxf(m, fmaxf(s[x + y], s[x + y + 8]));
                            m8[x] = m;
                        }
                        const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * sl2;  // sl2 > 0
                        if (j == 0) {
                            m_used = mx;
                        } else if (__any_sync(0xffffffffu, mx > m_used + RESCALE_LOG2)) {
                            const float m_new = fmaxf(mx, m_used);
                            alpha = (m_used == -INFINITY) ? 1.f : ex2(m_used - m_new);
                            m_used = m_new;
                            rescale = true;
                        }
                    }
                    const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
                    const float2 sc2 = make_float2(sl2, sl2), nm2 = make_float2(neg_m, neg_m);
                    acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int x = 0; x < BN; x += 2) {
                        const float2 v = __ffma2_rn(make_float2(s[x], s[x + 1]), sc2, nm2);
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(ex2(v.x), ex2(v.y));
                        // the row sum adds the same rounded weights the PV product uses
                        acc = add_bf16x2_f32(acc, *reinterpret_cast<uint32_t*>(&h2));
                        packed[x / 2] = __uint_as_float(*reinterpret_cast<uint32_t*>(&h2));
                    }
                    // (!(x <= bound) also sends a NaN sum to the second pass)
                    if (full || !__any_sync(0xffffffffu, !(acc.x + acc.y <= 65536.f))) break;
                }
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) tmem_st16(sbuf + hh * 16, packed + hh * 16);  // P over S_t[0, 64)
                if (rescale) {
                    // S_t(g) was issued after PV_t(g - 1) on the in-order tensor pipe, so its
                    // completion means O_t already holds every earlier block of the piece
                    for (int c0 = 0; c0 < HD; c0 += 32) {
                        float o[32];
                        tmem_ld32(tmem + lane_base + TM_O + t * 128 + c0, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int x = 0; x < 32; ++x) o[x] *= alpha;
                        tmem_st32(tmem + lane_base + TM_O + t * 128 + c0, o);
                    }
                }
                l_sum = l_sum * alpha + (acc.x + acc.y);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(BAR_P + t));
            }
            if (!ok) break;
            // ------------------------------------------------------------ epilogue of the piece
            ok = __all_sync(0xffffffffu, mbar_wait(bar(BAR_DONE), q & 1, wait_ns) && !aborted(abort_flag));
            if (!ok) break;
            tc_fence_after();
            Item it;
            {
                int w2 = w_item;
                next_item(w2, a, it);
            }
            const int gr = (it.rb * 2 + t) * 128 + r;
            const bool row_ok = gr < a.R;
            const int node = row_ok ? gr / a.G : 0;
            const float inv = (row_ok && l_sum > 0.f) ? 1.f / l_sum : 0.f;
            const bool cut = it.jb > 0 || it.je < it.nb;
            __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.O) +
                                  (((size_t)it.b * a.Kmax + node) * a.Hq + it.kvh * a.G + gr % a.G) * HD;
            const int slot = cut ? cut_slot(it.jb == 0, (int)blockIdx.x) : 0;
            // cut partials are stored chunk-major: float4 chunk x of rows 0..127 side by side, so every
            // warp store here and every warp load of the merge covers 512 contiguous bytes
            for (int c0 = 0; c0 < HD; c0 += 32) {
                float o[32];
                tmem_ld32(tmem + lane_base + TM_O + t * 128 + c0, o);
                tmem_wait_ld();
                if (c0 == HD - 32) {
                    // O_t is in registers: the next piece's first PV may overwrite it
                    tc_fence_before();
                    mbar_arrive(bar(BAR_OFREE + t));
                }
                if (!row_ok) continue;
                if (!cut) {
#pragma unroll
                    for (int x = 0; x < 32; x += 16) {
                        uint32_t wd[8];
#pragma unroll
                        for (int y = 0; y < 8; ++y) {
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(o[x + 2 * y] * inv, o[x + 2 * y + 1] * inv);
                            wd[y] = *reinterpret_cast<uint32_t*>(&h2);
                        }
                        st_global_v8(orow + c0 + x, wd);  // O rows start 32-byte aligned (the launch checks O)
                    }
                } else {
                    float4* pcol = reinterpret_cast<float4*>(a.cut_o) + ((size_t)(slot * 2 + t) * (HD / 4) + c0 / 4) * 128 + r;
                    // eight chunks 128 float4 (2 KB) apart
                    st_global_v4<0>(pcol, o[0] * inv, o[1] * inv, o[2] * inv, o[3] * inv);
                    st_global_v4<2048>(pcol, o[4] * inv, o[5] * inv, o[6] * inv, o[7] * inv);
                    st_global_v4<4096>(pcol, o[8] * inv, o[9] * inv, o[10] * inv, o[11] * inv);
                    st_global_v4<6144>(pcol, o[12] * inv, o[13] * inv, o[14] * inv, o[15] * inv);
                    st_global_v4<8192>(pcol, o[16] * inv, o[17] * inv, o[18] * inv, o[19] * inv);
                    st_global_v4<10240>(pcol, o[20] * inv, o[21] * inv, o[22] * inv, o[23] * inv);
                    st_global_v4<12288>(pcol, o[24] * inv, o[25] * inv, o[26] * inv, o[27] * inv);
                    st_global_v4<14336>(pcol, o[28] * inv, o[29] * inv, o[30] * inv, o[31] * inv);
                }
            }
            if (cut) {
                // -------------------------------------------- a cut piece
                if (row_ok) a.cut_lse[((size_t)slot * 2 + t) * 128 + r] = m_used + log2f(l_sum);
                const int kb = (slot & 1) * 2 + t;  // one-shot barriers of this slot kind and tile
                mbar_arrive(bar(BAR_CUT + kb));
                int32_t* cnt = a.cut_cnt + (size_t)it.idx * 2 + t;
                // the pieces run in groups q_first..q_last, in each on the CTA of this row-tile pair
                const int q_first = it.g_start / s_S, q_last = (it.g_start + it.nb - 1) / s_S;
                if (r == 0) {
                    // every row of the tile is written (the barrier orders them before this thread's fence,
                    // which is cumulative): publish them device-wide, then count this piece in
                    int old = -1;
                    if (mbar_wait(bar(BAR_CUT + kb), 0, wait_ns)) {
                        __threadfence();
                        old = atomicAdd(cnt, 1);
                        __threadfence();
                    }
                    s_last[t] = old;
                    mbar_arrive(bar(BAR_CUTL + kb));
                }
                ok = __all_sync(0xffffffffu, mbar_wait(bar(BAR_CUTL + kb), 0, wait_ns) && !aborted(abort_flag));
                if (!ok) break;
                const int old = s_last[t];
                if (old < 0) {
                    ok = false;
                    break;
                }
                if (old > q_last - q_first) flag_status(a.status, GRAFT_STATUS_WORKSPACE);  // counter not zeroed
                if (old == q_last - q_first) {
                    // the last piece to arrive: every piece's partial is complete (each wrote, and its CTA
                    // fenced before counting it in); merge them into the bf16 output and leave the
                    // counter at zero.  Loads are issued in batches before they are used (one round trip
                    // per batch): every piece's log2-sum-exp, then two pieces' 32 columns at a time.
                    if (r == 0) *cnt = 0;
                    if (row_ok) merge_cut_pieces(a.cut_lse, a.cut_o, orow, q_first, q_last - q_first + 1, nrb2, it.rb, t, r);
                }
            }
            g0 += it.je - it.jb;
            ++q;
        }
        if (!ok && !aborted(abort_flag)) raise_abort(abort_flag, a.status);
    }
    // ---------------------------------------------------------------- teardown
    if (warp == 0 && lane == 0 && aborted(abort_flag)) {
        // loads still in flight write into this CTA's shared memory: wait for the last armed
        // phase of every stage (and the last Q load) before the CTA may exit
        if (q_issued > 0) mbar_wait(bar(BAR_Q), (q_issued - 1) & 1, kDrainNs);
        for (int st = 0; st < SK; ++st) {
            const int n = (k_issued - st + SK - 1) / SK;
            if (n > 0) mbar_wait(bar(BAR_KF + st), (n - 1) & 1, kDrainNs);
        }
        for (int st = 0; st < SV; ++st) {
            const int n = (v_issued - st + SV - 1) / SV;
            if (n > 0) mbar_wait(bar(BAR_VF + st), (n - 1) & 1, kDrainNs);
        }
    }
    if (warp == 1 && lane == 0) {
        // every issued MMA has completed before TMEM is released: on an abort the MMAs issued
        // since the last piece's DONE get a commit of their own
        if (aborted(abort_flag)) {
            mma_commit(bar(BAR_DONE));
            ++ndone;
        }
        if (ndone > 0) mbar_wait(bar(BAR_DONE), (ndone - 1) & 1, kTeardownNs);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool encode(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box) {
    auto enc = encoder();
    if (enc == nullptr) return false;
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace attn_tcs

int attn_tcs_launch(const AttnArgs& a, int ctas, cudaStream_t st) {
    using namespace attn_tcs;
    // one key chunk per request, at most MAX_ORDER requests, CTAs in whole groups of row-tile pairs
    if (a.nRB % 2 != 0 || ctas < 1 || a.nchunk != 1 || a.B > MAX_ORDER || ctas % (a.nRB / 2) != 0)
        return GRAFT_ERR_INVALID_ARG;
    Maps m;
    const cuuint64_t es = 2;
    // Q: (dim, head, node) over [B*Kmax][Hq][128]
    {
        cuuint64_t dims[3] = {HD, (cuuint64_t)a.Hq, (cuuint64_t)a.B * a.Kmax};
        cuuint64_t strides[2] = {HD * es, (cuuint64_t)a.Hq * HD * es};
        cuuint32_t box[3] = {64, (cuuint32_t)a.G, (cuuint32_t)(128 / a.G)};
        if (!encode(&m.q, a.Q, 3, dims, strides, box)) return GRAFT_ERR_CUDA;
    }
    // caches: (dim, kv head, position, request) over [B][Lcap][Hkv][128]
    {
        const cuuint64_t Lc = a.Lcap > 0 ? (cuuint64_t)a.Lcap : 1;
        cuuint64_t dims[4] = {HD, (cuuint64_t)a.Hkv, Lc, (cuuint64_t)a.B};
        cuuint64_t strides[3] = {HD * es, (cuuint64_t)a.Hkv * HD * es, Lc * a.Hkv * HD * es};
        cuuint32_t box[4] = {64, 1, (cuuint32_t)BN, 1};
        const void* kc = a.Kc ? a.Kc : a.Kt;  // an empty cache is never read
        const void* vc = a.Vc ? a.Vc : a.Vt;
        if (!encode(&m.kc, kc, 4, dims, strides, box)) return GRAFT_ERR_CUDA;
        if (!encode(&m.vc, vc, 4, dims, strides, box)) return GRAFT_ERR_CUDA;
    }
    // tree KV: (dim, kv head, node, request) over [B][Kmax][Hkv][128]; nodes >= Kmax read as zeros
    {
        cuuint64_t dims[4] = {HD, (cuuint64_t)a.Hkv, (cuuint64_t)a.Kmax, (cuuint64_t)a.B};
        cuuint64_t strides[3] = {HD * es, (cuuint64_t)a.Hkv * HD * es, (cuuint64_t)a.Kmax * a.Hkv * HD * es};
        cuuint32_t box[4] = {64, 1, (cuuint32_t)BN, 1};
        if (!encode(&m.kt, a.Kt, 4, dims, strides, box)) return GRAFT_ERR_CUDA;
        if (!encode(&m.vt, a.Vt, 4, dims, strides, box)) return GRAFT_ERR_CUDA;
    }
    static bool attr_set[64][2] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    const bool test_waits = a.wait_ns != kWaitNs;
    auto kernel = test_waits ? attn_tcs_kernel<true> : attn_tcs_kernel<false>;
    if (dev >= 0 && dev < 64 && !attr_set[dev][test_waits]) {
        if (!cuda_ok(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES)))
            return GRAFT_ERR_CUDA;
        attr_set[dev][test_waits] = true;
    }
    launch_pdl(kernel, dim3(ctas), dim3(NTHREADS), SMEM_BYTES, st, m, a);
    count_launches(1);
    return launch_status();
}

}  // namespace graft
