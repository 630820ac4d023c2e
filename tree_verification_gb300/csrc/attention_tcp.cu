// Tree-masked GQA attention on the 5th-generation tensor cores, persistent
// variant of the two-tile kernel (attention_tc.cu) for grids of several
// waves.
//
// Graft article, architecture paragraph: the hybrid tree is verified on the
// standard tree-attention path in one target forward; Graft abstract: large
// draft trees cost VRAM bandwidth and compute.  Each query row (tree node i,
// query head h) attends to its request's L prefix keys and to the tree keys
// in node i's ancestor-or-self mask, with KV head h / group.
//
// A work item is what one CTA of the two-tile kernel does: two 128-row tiles
// of one (request, KV head) against one key chunk.  Items are ordered
// longest request first and dealt to at most one CTA per SM in a snake order
// (round k gives item k P + p to CTA p when k is even, to CTA P - 1 - p when
// k is odd), which balances items of decreasing size.  A CTA runs its items
// back to back through one pipeline:
//   * K and V blocks of consecutive items flow through the same rings with
//     running stage and phase counters, so the first blocks of the next item
//     load while the current one finishes;
//   * the next item's Q tiles load as soon as the current item's last S
//     product has run (its K-release barrier);
//   * the epilogue reads O out of TMEM, lets the next item's first PV
//     overwrite it (an O-free barrier per tile) and writes the rows straight
//     from registers (bf16 output rows, or fp32 partial rows and their
//     log2-sum-exp for the merge kernel), so it overlaps the next item's
//     first S product and softmax instead of staging through the rings.
// Everything else (TMEM layout, masking, lazy rescale) is the two-tile
// kernel's, except:
//   * the MMA issuer is a single thread with running ring counters, and it
//     tests the barrier of the next group of products (non-blocking) just
//     before the last two products of the current group: the tensor pipe
//     queues hardly any products ahead, so the issuer's own time between
//     products, waits included, is pipe idle time;
//   * the two tiles' softmax warps run their exponentials freely (no
//     turn-taking hand-off between the tiles);
//   * tile 0's softmax warps zero a ragged block's V rows past the chunk end
//     before they signal P_0.
//
// Every mbarrier wait is bounded; on timeout the CTA raises
// GRAFT_STATUS_TIMEOUT, stops issuing work, drains what it issued (again
// with a bound) and frees its TMEM before returning.
//
// This kernel deals whole items; attention_tcs.cu runs the same pipeline with
// the key blocks split evenly over the CTAs.  They are separate kernels
// because one kernel holding both schedules measured 13-18% slower per key
// block: the extra code around the hot loops doubled the warps' stalls on
// instruction fetch.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>

#include "attention.cuh"
#include "common.cuh"
#include "tc_ptx.cuh"

namespace graft {
namespace attn_tcp {

using namespace tc;

constexpr int HD = GRAFT_HEAD_DIM;
constexpr int BN = ATTN_TC_BLOCK_KEYS;  // keys per block
constexpr int SK = 2;                   // K ring depth
constexpr int SV = 3;                   // V ring depth
constexpr int NTHREADS = 320;
constexpr int MAX_ORDER = 256;          // requests ranked by length in shared memory
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
constexpr int N_BARS = BAR_OFREE + 2;
constexpr uint32_t OFF_MISC = OFF_BAR + N_BARS * 8;  // tmem slot, abort flag
constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

constexpr uint32_t TM_S = 0;    // + tile * 128
constexpr uint32_t TM_O = 256;  // + tile * 128
constexpr float RESCALE_LOG2 = 8.f;
constexpr uint64_t kWaitNs = 500000000ull;   // bound on any pipeline wait (the kernel runs for microseconds)
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

// One work item: both tiles of row pair rb of (request b, KV head kvh) against key chunk c.
struct Item {
    int b, kvh, rb, c;
    int k0, nb_prefix, nb, ragged_block, ragged_valid;
    bool skip, bad, direct;
};

// Item i in longest-request-first order: i = ((z * nchunk + c) * Hkv + kvh) * nrb2 + rb with z the
// rank of the request's length.
__device__ __forceinline__ Item make_item(const AttnArgs& a, const int* order, int i, int nrb2) {
    Item it;
    it.rb = i % nrb2;
    i /= nrb2;
    it.kvh = i % a.Hkv;
    i /= a.Hkv;
    it.c = i % a.nchunk;
    const int z = i / a.nchunk;
    it.b = order != nullptr ? order[z] : z;
    const int Lb = a.L[it.b];
    it.bad = Lb < 0 || Lb > a.Lcap;
    const int Cb = chunk_len(a, it.bad ? 0 : Lb);
    const int nck = (Lb > 0 && !it.bad) ? (Lb + Cb - 1) / Cb : 1;
    // a split request whose prefix leaves a chunk idle gives it the tree block
    const int tree_chunk = (nck > 1 && nck < a.nchunk) ? nck : nck - 1;
    it.skip = it.bad || it.c > tree_chunk;
    it.direct = nck == 1;
    it.k0 = it.c * Cb;
    const int k1 = it.bad ? it.k0 : max(it.k0, min(Lb, it.k0 + Cb));
    it.nb_prefix = (k1 - it.k0 + BN - 1) / BN;
    it.nb = it.skip ? 0 : it.nb_prefix + (it.c == tree_chunk ? 1 : 0);
    it.ragged_valid = (k1 - it.k0) % BN;
    it.ragged_block = it.ragged_valid != 0 ? it.nb_prefix - 1 : -1;
    return it;
}

// The snake deal: this CTA's k-th item, or -1 past the end.
__device__ __forceinline__ int item_index(int k, int n_items) {
    const int P = gridDim.x, p = blockIdx.x;
    const int i = k * P + ((k & 1) ? (P - 1 - p) : p);
    return i < n_items ? i : -1;
}

// A position (item, block) in this CTA's stream of blocks over its non-skipped items.
struct Cursor {
    int k;  // the item's place in this CTA's deal; -1 once past the last item
    Item it;
    int j;
};

__device__ __forceinline__ void seek_live(Cursor& cu, const AttnArgs& a, const int* order, int nrb2, int n_items) {
    for (;; ++cu.k) {
        const int i = item_index(cu.k, n_items);
        if (i < 0) {
            cu.k = -1;
            return;
        }
        cu.it = make_item(a, order, i, nrb2);
        if (!cu.it.skip) {
            cu.j = 0;
            return;
        }
    }
}

__device__ __forceinline__ void advance(Cursor& cu, const AttnArgs& a, const int* order, int nrb2, int n_items) {
    if (cu.k < 0) return;
    if (++cu.j < cu.it.nb) return;
    ++cu.k;
    seek_live(cu, a, order, nrb2, n_items);
}

// kTestWaits: pipeline waits bounded by a.wait_ns (the failure-path tests); otherwise by kWaitNs, a
// compile-time constant, so the production instantiation carries no run-time bound.
template <bool kTestWaits>
__global__ void __launch_bounds__(NTHREADS, 1)
attn_tcp_kernel(const __grid_constant__ Maps maps, AttnArgs a) {
    const uint64_t wait_ns = kTestWaits ? a.wait_ns : kWaitNs;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_order[MAX_ORDER];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + OFF_MISC);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + OFF_MISC + 4);
    auto bar = [&](int i) { return base + OFF_BAR + 8u * (uint32_t)i; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nrb2 = a.nRB / 2;  // row-tile pairs per (request, KV head); the launch needs nRB even
    const int n_items = a.B * a.nchunk * a.Hkv * nrb2;

    // Prologue that touches no global memory: it overlaps the previous kernel's tail.
    if (tid == 0) {
        for (int i = 0; i < N_BARS; ++i) {
            uint32_t cnt = 1;
            if (i == BAR_P || i == BAR_P + 1 || i == BAR_OFREE || i == BAR_OFREE + 1) cnt = 128;
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
    const bool ranked = a.B > 1 && a.B <= MAX_ORDER;
    if (ranked && tid < a.B) {
        const int li = a.L[tid];
        int rank = 0;
        for (int j = 0; j < a.B; ++j) {
            const int lj = a.L[j];
            rank += (lj > li) || (lj == li && j < tid);
        }
        s_order[rank] = tid;
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int* order = ranked ? s_order : nullptr;

    int k_issued = 0, v_issued = 0, q_issued = 0;  // blocks and Q pairs the producer has armed
    int ndone = 0;                   // DONE commits of the MMA issuer
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (lane 0)
        if (lane == 0) {
            auto load_q = [&](const Item& it) {
                ++q_issued;
                mbar_expect_tx(bar(BAR_Q), 2 * Q_TILE_BYTES);
                for (int t = 0; t < 2; ++t) {
                    const int nz = it.b * a.Kmax + (it.rb * 256 + t * 128) / a.G;
                    for (int h = 0; h < 2; ++h)
                        tma_load_3d(base + OFF_Q + t * Q_TILE_BYTES + h * (Q_TILE_BYTES / 2), &maps.q, bar(BAR_Q),
                                    h * 64, it.kvh * a.G, nz);
                }
            };
            auto load_block = [&](const Cursor& cu, const CUtensorMap* prefix_map, const CUtensorMap* tree_map,
                                  uint32_t dst, uint32_t full) {
                mbar_expect_tx(full, BLK_BYTES);
                for (int h = 0; h < 2; ++h) {
                    if (cu.j < cu.it.nb_prefix)
                        tma_load_4d(dst + h * BOX_BYTES, prefix_map, full, h * 64, cu.it.kvh, cu.it.k0 + cu.j * BN,
                                    cu.it.b);
                    else
                        tma_load_4d(dst + h * BOX_BYTES, tree_map, full, h * 64, cu.it.kvh, 0, cu.it.b);
                }
            };
            auto load_k = [&](Cursor& cu) {
                load_block(cu, &maps.kc, &maps.kt, base + OFF_K + (k_issued % SK) * BLK_BYTES,
                           bar(BAR_KF + k_issued % SK));
                ++k_issued;
                advance(cu, a, order, nrb2, n_items);
            };
            auto load_v = [&](Cursor& cu) {
                load_block(cu, &maps.vc, &maps.vt, base + OFF_V + (v_issued % SV) * BLK_BYTES,
                           bar(BAR_VF + v_issued % SV));
                ++v_issued;
                advance(cu, a, order, nrb2, n_items);
            };
            Cursor kc{0, Item{}, 0};
            seek_live(kc, a, order, nrb2, n_items);
            Cursor vc = kc, cc = kc;
            if (kc.k >= 0) load_q(kc.it);
            for (int s = 0; s < SK && kc.k >= 0; ++s) load_k(kc);
            for (int s = 0; s < SV && vc.k >= 0; ++s) load_v(vc);
            // Stages are released in the tensor pipe's order S_1(g), PV_1(g), S_1(g + 1), ..., so
            // one thread that waits for each release in turn never waits behind a later one.
            for (int g = 0; cc.k >= 0; ++g) {
                Cursor nx = cc;
                advance(nx, a, order, nrb2, n_items);
                const bool next_q = nx.k >= 0 && nx.j == 0;  // block g ends its item: the next Q follows
                if (kc.k >= 0 || next_q) {
                    if (!mbar_wait(bar(BAR_KE + g % SK), (g / SK) & 1, wait_ns)) {
                        raise_abort(abort_flag, a.status);
                        break;
                    }
                    if (aborted(abort_flag)) break;
                    // every S product of the item has run: its Q tiles are free
                    if (next_q) load_q(nx.it);
                    if (kc.k >= 0) load_k(kc);
                }
                if (vc.k >= 0) {
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
        // tcgen05.mma issue barely queues ahead of the tensor pipe, so every cycle this thread
        // spends between two products is a cycle the pipe idles: one thread runs the loop, with
        // the ring positions kept as running counters and no warp-wide votes.  (A second issuer
        // for the other tile, interleaving its products with these, measured slower.)
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
            // A group of eight products; just before its last two, a non-blocking test of the barrier
            // the next group needs is issued, so its latency overlaps the blocked issue of these
            // products; the blocking wait then runs only if the test came back false.  (Plain values,
            // no references: address-taken locals would live in local memory.)
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
            int q = 0;  // live items issued
            for (int k = 0; ok; ++k) {
                const int i = item_index(k, n_items);
                if (i < 0) break;
                const Item it = make_item(a, order, i, nrb2);
                if (it.skip) continue;
                ok = mbar_wait(bar(BAR_Q), q & 1, wait_ns) && !aborted(abort_flag) &&
                     mbar_wait(bar(BAR_KF + kst), kph, wait_ns);
                if (!ok) break;
                tc_fence_after();
                group_S(0, none);
                Pre vf{BAR_VF + vst, (uint32_t)vph};
                bool vf_ready = group_S(1, vf);
                for (int j = 0; j < it.nb && ok; ++j) {
                    // (tile 0's softmax warps zero a ragged block's V rows past the chunk end before
                    // they signal P_0, so PV_0 and PV_1, issued after that signal, read zeros there)
                    const bool more = j + 1 < it.nb;
                    ok = wait_pre(vf, vf_ready) && mbar_wait(bar(BAR_P), pph, wait_ns);
                    // the item's first PV overwrites O_t: the previous item's epilogue must have read it
                    if (ok && j == 0 && q > 0) ok = mbar_wait(bar(BAR_OFREE), (q - 1) & 1, wait_ns);
                    if (!ok) break;
                    tc_fence_after();
                    const Pre kf{BAR_KF + kst, (uint32_t)kph};
                    const Pre p1{BAR_P + 1, pph};
                    bool p1_ready;
                    if (more) {
                        const bool kf_ready = group_PV(0, j == 0, kf);
                        // this tile's next S right behind its PV: the other tile's softmax overlaps both
                        ok = wait_pre(kf, kf_ready);
                        if (!ok) break;
                        tc_fence_after();
                        p1_ready = group_S(0, p1);
                    } else {
                        p1_ready = group_PV(0, j == 0, p1);
                    }
                    ok = wait_pre(p1, p1_ready);
                    if (ok && j == 0 && q > 0) ok = mbar_wait(bar(BAR_OFREE + 1), (q - 1) & 1, wait_ns);
                    if (!ok) break;
                    tc_fence_after();
                    const int vst_next = vst + 1 == SV ? 0 : vst + 1;
                    const int vph_next = vst + 1 == SV ? vph ^ 1 : vph;
                    vf = Pre{BAR_VF + vst_next, (uint32_t)vph_next};
                    group_PV(1, j == 0, none);
                    vf_ready = more ? group_S(1, vf) : false;
                    vst = vst_next;
                    vph = vph_next;
                    pph ^= 1u;
                }
                // the item's MMAs (and everything before them) complete: its epilogue may read O
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
        const bool parts = a.nchunk > 1 && a.part_lse != nullptr;
        bool ok = true;
        int q = 0, g0 = 0;
        for (int k = 0; ok; ++k) {
            const int i = item_index(k, n_items);
            if (i < 0) break;
            // The block loop needs only the item's block counts; its coordinates are decoded again
            // for the epilogue (from i), so they hold no registers across the loop.
            int nb, nb_prefix, ragged_block, ragged_valid;
            uint64_t anc;
            {
                const Item it = make_item(a, order, i, nrb2);
                const int tile = it.rb * 2 + t;
                const size_t pbase = ((((size_t)it.b * a.Hkv + it.kvh) * a.nRB + tile) * a.nchunk + it.c) * 128;
                if (it.skip) {
                    if (it.bad && it.c == 0 && it.rb == 0 && it.kvh == 0 && t == 0 && r == 0)
                        flag_status(a.status, GRAFT_STATUS_LENGTH);
                    // a chunk past the request's keys contributes nothing to the merge
                    if (parts) a.part_lse[pbase + r] = -INFINITY;
                    continue;
                }
                // a request that fits one chunk writes its rows directly; the merge leaves them alone
                if (it.direct && parts) a.part_lse[pbase + r] = INFINITY;
                const int gr = tile * 128 + r;
                anc = gr < a.R ? a.mask[(size_t)it.b * a.Kmax + gr / a.G] : 0ull;
                nb = it.nb;
                nb_prefix = it.nb_prefix;
                ragged_block = it.ragged_block;
                ragged_valid = it.ragged_valid;
            }
            float m_used = -INFINITY, l_sum = 0.f;  // running max (log2 units) and row sum
            for (int j = 0; j < nb; ++j) {
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
                // An item's first block takes its maximum; a later block is first weighed against the
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
                        uint32_t w[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const int n = valid - 32 * x;
                            w[x] = n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
                        }
                        if (tree_blk) {
                            w[0] &= (uint32_t)anc;
                            w[1] &= (uint32_t)(anc >> 32);
                            w[2] = w[3] = 0u;
                        }
#pragma unroll
                        for (int x = 0; x < BN; ++x) s[x] = ((w[x >> 5] >> (x & 31)) & 1u) ? s[x] : -INFINITY;
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
                    // completion means O_t already holds every earlier block of the item
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
            // ------------------------------------------------------------ epilogue of the item
            ok = __all_sync(0xffffffffu, mbar_wait(bar(BAR_DONE), q & 1, wait_ns) && !aborted(abort_flag));
            if (!ok) break;
            tc_fence_after();
            const Item it = make_item(a, order, i, nrb2);
            const int tile = it.rb * 2 + t;
            const size_t pbase = ((((size_t)it.b * a.Hkv + it.kvh) * a.nRB + tile) * a.nchunk + it.c) * 128;
            const int gr = tile * 128 + r;
            const bool row_ok = gr < a.R;
            const int node = row_ok ? gr / a.G : 0;
            const float inv = (row_ok && l_sum > 0.f) ? 1.f / l_sum : 0.f;
            __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.O) +
                                  (((size_t)it.b * a.Kmax + node) * a.Hq + it.kvh * a.G + gr % a.G) * HD;
            float* prow = a.part_o + (pbase + r) * HD;
            for (int c0 = 0; c0 < HD; c0 += 32) {
                float o[32];
                tmem_ld32(tmem + lane_base + TM_O + t * 128 + c0, o);
                tmem_wait_ld();
                if (c0 == HD - 32) {
                    // O_t is in registers: the next item's first PV may overwrite it
                    tc_fence_before();
                    mbar_arrive(bar(BAR_OFREE + t));
                }
                if (!row_ok) continue;
                if (it.direct) {
#pragma unroll
                    for (int x = 0; x < 32; x += 16) {
                        uint32_t w[8];
#pragma unroll
                        for (int y = 0; y < 8; ++y) {
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(o[x + 2 * y] * inv, o[x + 2 * y + 1] * inv);
                            w[y] = *reinterpret_cast<uint32_t*>(&h2);
                        }
                        st_global_v8(orow + c0 + x, w);  // O rows start 32-byte aligned (the launch checks O)
                    }
                } else {
#pragma unroll
                    for (int x = 0; x < 32; x += 8) {
                        uint32_t w[8];
#pragma unroll
                        for (int y = 0; y < 8; ++y) w[y] = __float_as_uint(o[x + y] * inv);
                        st_global_v8(prow + c0 + x, w);
                    }
                }
            }
            if (!it.direct && row_ok) a.part_lse[pbase + r] = m_used + log2f(l_sum);
            g0 += nb;
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
        // since the last item's DONE get a commit of their own
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

}  // namespace attn_tcp

int attn_tcp_items(const AttnArgs& a) { return a.B * a.nchunk * a.Hkv * (a.nRB / 2); }

int attn_tcp_launch(const AttnArgs& a, int ctas, cudaStream_t st) {
    using namespace attn_tcp;
    if (a.nRB % 2 != 0 || ctas < 1) return GRAFT_ERR_INVALID_ARG;
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
    auto kernel = test_waits ? attn_tcp_kernel<true> : attn_tcp_kernel<false>;
    if (dev >= 0 && dev < 64 && !attr_set[dev][test_waits]) {
        if (!cuda_ok(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES)))
            return GRAFT_ERR_CUDA;
        attr_set[dev][test_waits] = true;
    }
    launch_pdl(kernel, dim3(ctas), dim3(NTHREADS), SMEM_BYTES, st, m, a);
    count_launches(1);
    const int rc = launch_status();
    if (rc != GRAFT_OK) return rc;
    return attn_combine_launch(a, st);
}

}  // namespace graft
