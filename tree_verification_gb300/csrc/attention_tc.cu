// Tree-masked GQA attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Graft article, architecture paragraph: the hybrid tree is verified on the
// standard tree-attention path in one target forward; Graft abstract: large
// draft trees cost VRAM bandwidth and compute.  Each query row (tree node i,
// query head h) attends to its request's L prefix keys and to the tree keys
// in node i's ancestor-or-self mask, with KV head h / group.
//
// One CTA computes two 128-row tiles of query rows (all query heads of one
// KV head for 256 / group tree nodes) against one key chunk, in 128-key
// blocks: every K/V byte brought into shared memory feeds 256 rows.
//
// Warp roles (10 warps):
//   warp 0      TMA producer (one lane): both Q tiles, then K blocks into a
//               2-stage ring and V blocks into a 3-stage ring (128-byte
//               swizzled boxes of 128 keys x 64 dims); a K stage is released
//               once both tiles' S products have run, a V stage once both
//               tiles' PV products have run
//   warp 1      owns the TMEM allocation (512 columns); MMA issuer (one
//               thread): S_t = Q_t K^T, O_t += P_t V.  The two tiles
//               ping-pong: as soon as tile t's P arrives its PV and its next
//               S are issued, so the tensor pipe works on one tile while the
//               other tile's softmax runs.  tcgen05.mma issue hardly queues
//               ahead of the pipe, so the issuer keeps its own time between
//               products short: the barrier the next group of products needs
//               is tested (non-blocking) just before the last two products
//               of the current group
//   warps 2-5   softmax + epilogue of tile 0 (one row per thread; warp w
//               reaches TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31); they also
//               zero a ragged block's V rows before they signal P_0
//   warps 6-9   softmax + epilogue of tile 1
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512).
// Softmax overwrites the first 64 columns of S_t with P_t as packed bf16
// pairs; the PV MMA takes that as its A operand straight from TMEM, so P
// never touches shared memory.  S_t(j + 1) is issued after PV_t(j) on the
// same in-order tensor pipe, so it cannot overwrite P_t(j) early, and its
// completion also certifies that O_t holds every block before j + 1.
//
// Softmax keeps a per-row running maximum that is only raised (and O
// rescaled) when a block's maximum exceeds it by more than 2^8, so the
// rescale of O in TMEM is rare; probabilities are then bounded by 256, which
// bf16 P and fp32 sums carry without loss of range.  The row sum adds the
// bf16-rounded probabilities, the same values the PV product consumes.
// Masked keys (ragged chunk tail, tree keys outside the ancestor mask) get
// probability 0, and the V rows of a ragged tail are zeroed in shared memory
// so stale cache rows cannot inject NaN.
//
// The epilogue stages each tile's rows through the freed K/V ring memory and
// writes them out along contiguous rows.
//
// Every mbarrier wait is bounded; on timeout the CTA raises
// GRAFT_STATUS_TIMEOUT in the status word, stops issuing work, drains what
// it issued (again with a bound) and frees its TMEM before returning.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>

#include "attention.cuh"
#include "common.cuh"
#include "tc_ptx.cuh"

namespace graft {
namespace attn_tc {

using namespace tc;

constexpr int HD = GRAFT_HEAD_DIM;
constexpr int BN = ATTN_TC_BLOCK_KEYS;  // keys per block
#ifndef ATTN_K_STAGES
#define ATTN_K_STAGES 2
#define ATTN_V_STAGES 3
#endif
constexpr int SK = ATTN_K_STAGES;       // K ring depth
constexpr int SV = ATTN_V_STAGES;       // V ring depth
constexpr int NTHREADS = 320;
constexpr uint32_t BOX_BYTES = BN * 64 * 2;             // one box: 128 keys (or rows) x 64 dims bf16
constexpr uint32_t BLK_BYTES = 2 * BOX_BYTES;           // one K or V block (128 keys x 128 dims)
constexpr uint32_t Q_TILE_BYTES = 2 * 128 * 64 * 2;     // 128 rows x 128 dims
// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + 2 * Q_TILE_BYTES;
constexpr uint32_t OFF_V = OFF_K + SK * BLK_BYTES;
constexpr uint32_t OFF_BAR = OFF_V + SV * BLK_BYTES;
constexpr uint32_t OFF_STAGE = OFF_K;  // epilogue staging reuses the rings once every MMA has run
// barriers
constexpr int BAR_Q = 0;              // Q tiles landed
constexpr int BAR_KF = 1;             // [SK] K block landed
constexpr int BAR_KE = BAR_KF + SK;   // [SK] K block consumed by both S products
constexpr int BAR_VF = BAR_KE + SK;   // [SV] V block landed
constexpr int BAR_VE = BAR_VF + SV;   // [SV] V block consumed by both PV products
constexpr int BAR_S = BAR_VE + SV;    // [tile] S_t ready in TMEM
constexpr int BAR_P = BAR_S + 2;      // [tile] P_t written to TMEM (128 arrivals)
constexpr int BAR_DONE = BAR_P + 2;   // every MMA completed (one-shot)
constexpr int BAR_EPI = BAR_DONE + 1; // [tile] staging written (128 arrivals, one-shot)
constexpr int BAR_ODONE = BAR_EPI + 2; // O_0 complete: tile 0's last PV ran (one-shot)
constexpr int N_BARS = BAR_ODONE + 1;
constexpr uint32_t OFF_MISC = OFF_BAR + N_BARS * 8;  // tmem slot, abort flag
constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(2 * 128 * 128 * 4 <= (SK + SV) * BLK_BYTES, "staging of both tiles fits in the rings");

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

// kTestWaits: pipeline waits bounded by a.wait_ns (the failure-path tests); otherwise by kWaitNs, a
// compile-time constant, so the production instantiation carries no run-time bound.
template <bool kTestWaits>
__global__ void __launch_bounds__(NTHREADS, 1)
attn_tc_kernel(const __grid_constant__ Maps maps, AttnArgs a) {
    const uint64_t wait_ns = kTestWaits ? a.wait_ns : kWaitNs;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + OFF_MISC);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + OFF_MISC + 4);
    auto bar = [&](int i) { return base + OFF_BAR + 8u * (uint32_t)i; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nrb2 = (a.nRB + 1) / 2;           // CTAs (pairs of 128-row tiles) per (request, KV head)
    const int rb = blockIdx.x % nrb2;
    const int kvh = blockIdx.x / nrb2;
    const int c = blockIdx.y;
    int b = blockIdx.z;  // remapped below to the request this CTA serves
    const int ntile = (2 * rb + 1 < a.nRB) ? 2 : 1;  // the last pair of an odd tile count has one

    // Prologue: it overlaps the previous kernel's tail, so it reads nothing it relies on from global
    // memory (the L2 warm-up below only takes a hint from it).
    if (tid == 0) {
        for (int i = 0; i < N_BARS; ++i) {
            uint32_t cnt = 1;
            if (i == BAR_P || i == BAR_P + 1 || i == BAR_EPI || i == BAR_EPI + 1)
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
        if (a.B == 1) {
            // L2 warm-up while the previous kernel finishes: this CTA's Q tiles and first K and V
            // block, placed by the request's length as it reads now.  A prefetch hands no data to the
            // CTA, and L2 is where every write lands, so a length or cache the previous kernel is still
            // writing costs at most a wasted prefetch; the loads proper follow the wait.  (Warming
            // three blocks per CTA measured slower: more DRAM traffic than the previous kernel's tail
            // hides.)
            const int Lh = a.L[0];
            const int k0 = c * chunk_len(a, Lh > 0 && Lh <= a.Lcap ? Lh : 0);
            if (Lh > 0 && Lh <= a.Lcap && k0 < Lh) {
                for (int t = 0; t < ntile; ++t)
                    for (int h = 0; h < 2; ++h)
                        tma_prefetch_l2_3d(&maps.q, h * 64, kvh * a.G, (rb * 256 + t * 128) / a.G);
                for (int h = 0; h < 2; ++h) {
                    tma_prefetch_l2_4d(&maps.kc, h * 64, kvh, k0, 0);
                    tma_prefetch_l2_4d(&maps.vc, h * 64, kvh, k0, 0);
                }
            }
        }
    }
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(base + OFF_MISC, 512);
        tmem_relinquish();
        tc_fence_before();
    }
    griddep_wait();
    griddep_launch_dependents();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Longest-first dispatch: CTAs launch in blockIdx.z order, so z maps to the z-th longest
    // request (ties to the lower index) and short requests fill the last wave.
    if (a.B > 1 && a.B <= NTHREADS) {
        __shared__ int s_req;
        if (tid < a.B) {
            const int li = a.L[tid];
            int rank = 0;
            for (int j = 0; j < a.B; ++j) {
                const int lj = a.L[j];
                rank += (lj > li) || (lj == li && j < tid);
            }
            if (rank == (int)blockIdx.z) s_req = tid;
        }
        __syncthreads();
        b = s_req;
    }
    const int Lb = a.L[b];
    const bool bad_len = Lb < 0 || Lb > a.Lcap;
    const int Cb = chunk_len(a, bad_len ? 0 : Lb);
    const int nck = (Lb > 0 && !bad_len) ? (Lb + Cb - 1) / Cb : 1;
    // A split request whose prefix leaves a chunk CTA idle gives it the tree block, so the last
    // prefix chunk does not carry one block more than the others.
    const int tree_chunk = (nck > 1 && nck < a.nchunk) ? nck : nck - 1;
    if (bad_len || c > tree_chunk) {  // uniform over the CTA
        if (bad_len && tid == 0 && c == 0 && rb == 0 && kvh == 0) flag_status(a.status, GRAFT_STATUS_LENGTH);
        for (int t = 0; t < ntile; ++t) mark_partial(a, b, kvh, rb * 2 + t, c, -INFINITY);
        if (warp == 1) tmem_dealloc(tmem, 512);
        return;
    }
    if (nck == 1)
        for (int t = 0; t < ntile; ++t) mark_partial(a, b, kvh, rb * 2 + t, 0, INFINITY);
    const int k0 = c * Cb;
    const int k1 = max(k0, min(Lb, k0 + Cb));
    const int nb_prefix = (k1 - k0 + BN - 1) / BN;
    const bool has_tree = (c == tree_chunk);
    const int nb = nb_prefix + (has_tree ? 1 : 0);
    const int ragged_block = ((k1 - k0) % BN) != 0 ? nb_prefix - 1 : -1;
    const int ragged_valid = (k1 - k0) % BN;

    int k_issued = 0, v_issued = 0;  // blocks the producer lanes have armed
    auto load_block = [&](int j, const CUtensorMap* prefix_map, const CUtensorMap* tree_map, uint32_t dst,
                          uint32_t full) {
        mbar_expect_tx(full, BLK_BYTES);
        for (int h = 0; h < 2; ++h) {
            if (j < nb_prefix)
                tma_load_4d(dst + h * BOX_BYTES, prefix_map, full, h * 64, kvh, k0 + j * BN, b);
            else
                tma_load_4d(dst + h * BOX_BYTES, tree_map, full, h * 64, kvh, 0, b);
        }
    };
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (lane 0)
        // Q tiles, then K and V blocks in the order their stages free up.  Stages are released
        // in the tensor pipe's order S_1(0), PV_1(0), S_1(1), PV_1(1), ..., so one thread that
        // waits for each release in turn never waits behind a later one.
        if (lane == 0) {
            mbar_expect_tx(bar(BAR_Q), ntile * Q_TILE_BYTES);
            for (int t = 0; t < ntile; ++t) {
                const int nz = b * a.Kmax + (rb * 256 + t * 128) / a.G;
                for (int h = 0; h < 2; ++h)
                    tma_load_3d(base + OFF_Q + t * Q_TILE_BYTES + h * (Q_TILE_BYTES / 2), &maps.q, bar(BAR_Q),
                                h * 64, kvh * a.G, nz);
            }
            auto load_k = [&](int j) {
                load_block(j, &maps.kc, &maps.kt, base + OFF_K + (j % SK) * BLK_BYTES, bar(BAR_KF + j % SK));
                ++k_issued;
            };
            auto load_v = [&](int j) {
                load_block(j, &maps.vc, &maps.vt, base + OFF_V + (j % SV) * BLK_BYTES, bar(BAR_VF + j % SV));
                ++v_issued;
            };
            for (int j = 0; j < SK || j < SV; ++j) {
                if (j < SK && j < nb) load_k(j);
                if (j < SV && j < nb) load_v(j);
            }
            for (int i = 0; i < nb; ++i) {
                // K(i + SK) reuses the stage S_1(i) released; V(i + SV) the one PV_1(i) released
                if (i + SK < nb) {
                    if (!mbar_wait(bar(BAR_KE + i % SK), (i / SK) & 1, wait_ns)) {
                        raise_abort(abort_flag, a.status);
                        break;
                    }
                    if (aborted(abort_flag)) break;
                    load_k(i + SK);
                }
                if (i + SV < nb) {
                    if (!mbar_wait(bar(BAR_VE + i % SV), (i / SV) & 1, wait_ns)) {
                        raise_abort(abort_flag, a.status);
                        break;
                    }
                    if (aborted(abort_flag)) break;
                    load_v(i + SV);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (lane 0 alone)
        // tcgen05.mma issue hardly queues ahead of the tensor pipe, so every cycle this thread
        // spends between two products, waits included, is a cycle the pipe idles: one thread runs
        // the loop, and the barrier the next group of products needs is tested (non-blocking)
        // just before the last two products of the current group, so the blocking wait runs only
        // when that test came back false.
        if (lane == 0) {
            const uint32_t idS = idesc_bf16(128, BN, false, false);
            const uint32_t idO = idesc_bf16(128, HD, false, true);
            // Descriptors are built once; each MMA adds a byte offset (in 16-byte units) to the
            // start-address field, which sits in the low bits and cannot carry out of them here
            // (every shared-memory address is below 256 KB).
            const uint64_t q_desc = sdesc_sw128(base + OFF_Q, 16, 1024);
            const uint64_t k_desc = sdesc_sw128(base + OFF_K, 16, 1024);
            const uint64_t v_desc = sdesc_sw128(base + OFF_V, BOX_BYTES, 1024);
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
            // S_t(jj) = Q_t K(jj)^T into S_t; the last tile's product releases K(jj)
            auto group_S = [&](int t, int jj, Pre nxt) -> bool {
                bool ready = false;
                const uint64_t kd = k_desc + (((jj % SK) * BLK_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    if (kk == HD / 16 - 2) ready = test_pre(nxt);
                    const uint32_t off = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
                    const uint32_t qoff = t * Q_TILE_BYTES + (kk >> 2) * (Q_TILE_BYTES / 2) + (kk & 3) * 32;
                    mma_bf16_ss(tmem + TM_S + t * 128, q_desc + (qoff >> 4), kd + (off >> 4), idS, kk > 0);
                }
                mma_commit(bar(BAR_S + t));
                if (t == ntile - 1) mma_commit(bar(BAR_KE + jj % SK));
                return ready;
            };
            // O_t += P_t V(j); the last tile's product releases V(j)
            auto group_PV = [&](int t, int j, Pre nxt) -> bool {
                bool ready = false;
                const uint32_t p = tmem + TM_S + t * 128;  // P_t as packed bf16 pairs
                const uint64_t vd = v_desc + (((j % SV) * BLK_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    if (kk == BN / 16 - 2) ready = test_pre(nxt);
                    mma_bf16_ts(tmem + TM_O + t * 128, p + kk * 8, vd + ((kk * 2048) >> 4), idO, j > 0 || kk > 0);
                }
                if (t == ntile - 1) mma_commit(bar(BAR_VE + j % SV));
                return ready;
            };
            bool ok = mbar_wait(bar(BAR_Q), 0, wait_ns) && (nb == 0 || mbar_wait(bar(BAR_KF), 0, wait_ns));
            Pre vf{BAR_VF, 0u};
            bool vf_ready = false;
            if (ok && nb > 0) {
                tc_fence_after();
                if (ntile == 2) group_S(0, 0, none);
                vf_ready = group_S(ntile - 1, 0, vf);
            }
            // (tile 0's softmax warps zero a ragged block's V rows past the chunk end before they
            // signal P_0, so every PV of that block, issued after that signal, reads zeros there)
            for (int j = 0; j < nb && ok; ++j) {
                const bool more = j + 1 < nb;
                ok = wait_pre(vf, vf_ready) && mbar_wait(bar(BAR_P), j & 1, wait_ns) && !aborted(abort_flag);
                if (!ok) break;
                tc_fence_after();
                const Pre kf{BAR_KF + (j + 1) % SK, (uint32_t)(((j + 1) / SK) & 1)};
                const Pre p1{BAR_P + 1, (uint32_t)(j & 1)};
                const Pre vn{BAR_VF + (j + 1) % SV, (uint32_t)(((j + 1) / SV) & 1)};
                if (ntile == 2) {
                    bool p1_ready;
                    if (more) {
                        const bool kf_ready = group_PV(0, j, kf);
                        // this tile's next S right behind its PV: the other tile's softmax overlaps both
                        ok = wait_pre(kf, kf_ready);
                        if (!ok) break;
                        tc_fence_after();
                        p1_ready = group_S(0, j + 1, p1);
                    } else {
                        p1_ready = group_PV(0, j, p1);
                        mma_commit(bar(BAR_ODONE));  // tile 0's epilogue may start
                    }
                    ok = wait_pre(p1, p1_ready);
                    if (!ok) break;
                    tc_fence_after();
                    group_PV(1, j, none);
                    vf_ready = more ? group_S(1, j + 1, vn) : false;
                } else if (more) {
                    const bool kf_ready = group_PV(0, j, kf);
                    ok = wait_pre(kf, kf_ready);
                    if (!ok) break;
                    tc_fence_after();
                    vf_ready = group_S(0, j + 1, vn);
                } else {
                    group_PV(0, j, none);
                    mma_commit(bar(BAR_ODONE));
                }
                vf = vn;
            }
            if (!ok && !aborted(abort_flag)) raise_abort(abort_flag, a.status);
            mma_commit(bar(BAR_DONE));
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int t = (warp - 2) >> 2;
        const int quad = warp & 3;
        const int r = quad * 32 + lane;  // row within the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const int gr = rb * 256 + t * 128 + r;
        const bool row_ok = t < ntile && gr < a.R;
        const int node = row_ok ? gr / a.G : 0;
        const uint64_t anc = row_ok ? a.mask[(size_t)b * a.Kmax + node] : 0ull;
        const float sl2 = a.scale * 1.4426950408889634f;
        float m_used = -INFINITY, l_sum = 0.f;  // running max (log2 units) and row sum
        bool ok = true;
        const uint32_t sbuf = tmem + lane_base + TM_S + t * 128;
        for (int j = 0; j < nb && t < ntile; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(BAR_S + t), j & 1, wait_ns) && !aborted(abort_flag));
            if (!ok) break;
            tc_fence_after();
            if (t == 0 && j == ragged_block) {
                // zero the V rows past the chunk end (both 64-dim boxes) before PV reads them: the
                // block's keys there are masked, but the cache rows may hold non-finite garbage
                ok = __all_sync(0xffffffffu, mbar_wait(bar(BAR_VF + j % SV), (j / SV) & 1, wait_ns));
                if (!ok) break;
                uint8_t* v0 = gbase + OFF_V + (j % SV) * BLK_BYTES;
                for (int x = r; x < (BN - ragged_valid) * 16; x += 128) {
                    const int rr = ragged_valid + x / 16, c16 = x % 16;
                    *reinterpret_cast<uint4*>(v0 + (c16 >= 8 ? BOX_BYTES : 0) + rr * 128 + (c16 & 7) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            float s[BN];
#pragma unroll
            for (int q = 0; q < BN / 32; ++q) tmem_ld32(sbuf + q * 32, s + q * 32);
            tmem_wait_ld();
            const bool tree_blk = j >= nb_prefix;
            if (tree_blk || j == ragged_block) {
                // only the ragged tail and the tree block need masking: keep-bits for the
                // block's keys as four 32-bit words (tree keys are < 64, in the ancestor mask)
                const int valid = tree_blk ? a.Kmax : ragged_valid;
                uint32_t w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int n = valid - 32 * q;
                    w[q] = n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
                }
                if (tree_blk) {
                    w[0] &= (uint32_t)anc;
                    w[1] &= (uint32_t)(anc >> 32);
                    w[2] = w[3] = 0u;
                }
#pragma unroll
                for (int i = 0; i < BN; ++i) s[i] = ((w[i >> 5] >> (i & 31)) & 1u) ? s[i] : -INFINITY;
            }
            // block maximum by a tree of pairwise maxima (short dependency chains)
            float m8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float m = fmaxf(s[i], s[i + 8]);
#pragma unroll
                for (int k = 16; k < BN; k += 16) m = fmaxf(m, fmaxf(s[i + k], s[i + k + 8]));
                m8[i] = m;
            }
            const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                   fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * sl2;  // sl2 > 0
            // raise the running maximum of the rows that need it; their O and row sum are
            // rescaled by 2^(m_used - m_new) below, once the S values are no longer live
            float alpha = 1.f;
            bool rescale = false;
            if (j == 0) {
                m_used = mx;
            } else if (__any_sync(0xffffffffu, mx > m_used + RESCALE_LOG2)) {
                const float m_new = fmaxf(mx, m_used);
                alpha = (m_used == -INFINITY) ? 1.f : ex2(m_used - m_new);
                m_used = m_new;
                rescale = true;
            }
            const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
            const float2 sc2 = make_float2(sl2, sl2), nm2 = make_float2(neg_m, neg_m);
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
                float packed[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float2 x = __ffma2_rn(make_float2(s[hh * 32 + i], s[hh * 32 + i + 1]), sc2, nm2);
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(ex2(x.x), ex2(x.y));
                    // the row sum adds the same rounded weights the PV product uses
                    acc = add_bf16x2_f32(acc, *reinterpret_cast<uint32_t*>(&h2));
                    packed[i / 2] = __uint_as_float(*reinterpret_cast<uint32_t*>(&h2));
                }
                tmem_st16(sbuf + hh * 16, packed);  // P over the first 64 columns of S_t
            }
            if (rescale) {
                // S_t(j) was issued after PV_t(j - 1) on the in-order tensor pipe, so its
                // completion means O_t already holds every earlier block; PV_t(j) waits for P_t(j)
                for (int c0 = 0; c0 < HD; c0 += 32) {
                    float o[32];
                    tmem_ld32(tmem + lane_base + TM_O + t * 128 + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= alpha;
                    tmem_st32(tmem + lane_base + TM_O + t * 128 + c0, o);
                }
            }
            l_sum = l_sum * alpha + (acc.x + acc.y);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(BAR_P + t));
        }
        if (!ok && !aborted(abort_flag)) raise_abort(abort_flag, a.status);
        // ------------------------------------------------------------ epilogue
        if (t < ntile) {
            if (ok && nb > 0) {
                // the tile's last PV has completed (one-shot barriers: no phase ambiguity); tile 0 needs
                // only its own (every S product, the K ring's last reader, ran before it), tile 1 every
                // product (its rows are staged over the V ring)
                ok = __all_sync(0xffffffffu, mbar_wait(bar(t == 0 ? BAR_ODONE : BAR_DONE), 0, wait_ns));
                if (!ok) raise_abort(abort_flag, a.status);
            }
            const bool direct = (nck == 1);
            const float inv = (row_ok && l_sum > 0.f) ? 1.f / l_sum : 0.f;
            uint8_t* stile = gbase + OFF_STAGE + t * (128 * 512);
            if (ok) {
                tc_fence_after();
                // stage this thread's row, 16-byte chunks permuted by the row index so a warp's
                // 32 rows spread over all banks
                uint8_t* srow = stile + r * (direct ? 256 : 512);
                for (int c0 = 0; c0 < HD; c0 += 32) {
                    float o[32];
                    tmem_ld32(tmem + lane_base + TM_O + t * 128 + c0, o);
                    tmem_wait_ld();
                    if (direct) {
#pragma unroll
                        for (int i = 0; i < 32; i += 8) {
                            uint4 v;
                            __nv_bfloat162 x0 = __floats2bfloat162_rn(o[i] * inv, o[i + 1] * inv);
                            __nv_bfloat162 x1 = __floats2bfloat162_rn(o[i + 2] * inv, o[i + 3] * inv);
                            __nv_bfloat162 x2 = __floats2bfloat162_rn(o[i + 4] * inv, o[i + 5] * inv);
                            __nv_bfloat162 x3 = __floats2bfloat162_rn(o[i + 6] * inv, o[i + 7] * inv);
                            v.x = *reinterpret_cast<uint32_t*>(&x0);
                            v.y = *reinterpret_cast<uint32_t*>(&x1);
                            v.z = *reinterpret_cast<uint32_t*>(&x2);
                            v.w = *reinterpret_cast<uint32_t*>(&x3);
                            const int chunk = (c0 + i) / 8;  // 0..15
                            *reinterpret_cast<uint4*>(srow + ((chunk ^ (r & 15)) << 4)) = v;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const int chunk = (c0 + i) / 4;  // 0..31
                            *reinterpret_cast<float4*>(srow + ((chunk ^ (r & 31)) << 4)) =
                                make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
                        }
                    }
                }
            }
            mbar_arrive(bar(BAR_EPI + t));
            const bool staged = __all_sync(0xffffffffu, mbar_wait(bar(BAR_EPI + t), 0, wait_ns));
            if (!staged) {
                raise_abort(abort_flag, a.status);
                ok = false;
            }
            if (ok) {
                // write the tile out along contiguous rows; 128 threads of this tile
                const int tile = rb * 2 + t;  // 128-row tile index within (b, kvh)
                if (direct) {
                    for (int k = r; k < 128 * 16; k += 128) {
                        const int row = k >> 4, cc = k & 15;
                        const int g = tile * 128 + row;
                        if (g >= a.R) continue;
                        const int nd = g / a.G, hh = kvh * a.G + g % a.G;
                        const uint4 v = *reinterpret_cast<const uint4*>(stile + row * 256 + ((cc ^ (row & 15)) << 4));
                        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.O) +
                                             (((size_t)b * a.Kmax + nd) * a.Hq + hh) * HD + cc * 8;
                        *reinterpret_cast<uint4*>(dst) = v;
                    }
                } else {
                    const size_t pbase = ((((size_t)b * a.Hkv + kvh) * a.nRB + tile) * a.nchunk + c) * 128;
                    float* dst = a.part_o + pbase * HD;
                    for (int k = r; k < 128 * 32; k += 128) {
                        const int row = k >> 5, cc = k & 31;
                        const float4 v = *reinterpret_cast<const float4*>(stile + row * 512 + ((cc ^ (row & 31)) << 4));
                        *reinterpret_cast<float4*>(dst + row * HD + cc * 4) = v;
                    }
                    if (row_ok) a.part_lse[pbase + r] = m_used + log2f(l_sum);
                }
            }
        }
    }
    // ---------------------------------------------------------------- teardown
    if (warp == 0 && lane == 0 && aborted(abort_flag)) {
        // loads still in flight write into this CTA's shared memory: the producer waits for the
        // last armed phase of every stage it used (and the Q load) before the CTA may exit
        mbar_wait(bar(BAR_Q), 0, kDrainNs);
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
        // every issued MMA has completed before TMEM is released
        mbar_wait(bar(BAR_DONE), 0, kTeardownNs);
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

}  // namespace attn_tc

bool attn_tc_supported(int G) { return G >= 1 && G <= 128 && (128 % G) == 0; }

int attn_tc_launch(const AttnArgs& a, cudaStream_t st) {
    using namespace attn_tc;
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
    auto kernel = test_waits ? attn_tc_kernel<true> : attn_tc_kernel<false>;
    if (dev >= 0 && dev < 64 && !attr_set[dev][test_waits]) {
        if (!cuda_ok(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES)))
            return GRAFT_ERR_CUDA;
        attr_set[dev][test_waits] = true;
    }
    launch_pdl(kernel, dim3(((a.nRB + 1) / 2) * a.Hkv, a.nchunk, a.B), dim3(NTHREADS), SMEM_BYTES, st, m, a);
    count_launches(1);
    const int rc = launch_status();
    if (rc != GRAFT_OK) return rc;
    return attn_combine_launch(a, st);
}

}  // namespace graft
