// Tree-masked GQA attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Graft article, architecture paragraph: the hybrid tree is verified on the
// standard tree-attention path in one target forward; Graft abstract: large
// draft trees cost VRAM bandwidth and compute.  Each query row (tree node i,
// query head h) attends to its request's L prefix keys and to the tree keys
// in node i's ancestor-or-self mask, with KV head h / group.
//
// One-tile variant: one CTA computes one 128-row tile of query rows (all
// query heads of one KV head for 128 / group tree nodes) against one key
// chunk, in 128-key blocks.  It suits short chunks (small batches, short
// prefixes: many CTAs with few blocks each), where its shorter prologue
// beats the two-tile kernel of attention_tc.cu, whose CTAs share each K/V
// block between two tiles.
//
// Warp roles (8 warps):
//   warp 0      TMA producer: the Q tile once, then K blocks into a 3-stage
//               ring (128-byte swizzled boxes of 128 keys x 64 dims); a K
//               stage is released as soon as its S product has run
//   warp 3      TMA producer: V blocks into their own 3-stage ring, a stage
//               released once its PV product has run
//   warp 1      MMA issuer (one thread): S = Q K^T with both operands in
//               shared memory, then O += P V with P read from TMEM;
//               shared-memory descriptors are built once and offset per MMA;
//               the barrier the next group of products needs is tested
//               (non-blocking) before the last two products of the current
//               group, since tcgen05.mma issue hardly queues ahead of the pipe
//   warp 2      owns the TMEM allocation (512 columns)
//   warps 4-7   softmax + epilogue (TMEM lanes 0-127, one query row per
//               thread); they zero a ragged block's V rows before its P
// TMEM columns: S/P double buffer [0,128) and [128,256), O [256,384).  The
// first S product issues as soon as the Q tile and the first K block have
// landed: Q is read by the tensor core from shared memory, which measured
// faster per MMA than a TMEM A operand at this shape and needs no copy
// before the first product.  Softmax overwrites the first 64 columns of its S buffer with P as packed bf16
// pairs; the PV MMA takes that as its A operand straight from TMEM, so P
// never touches shared memory.
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
// The epilogue stages the tile's rows through the freed K/V ring memory and
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
namespace attn_tc1 {

using namespace tc;

constexpr int HD = GRAFT_HEAD_DIM;
constexpr int BN = ATTN_TC_BLOCK_KEYS;  // keys per block
constexpr int SK = 3;                   // K ring depth
constexpr int SV = 3;                   // V ring depth
constexpr int NTHREADS = 256;
constexpr uint32_t BOX_BYTES = BN * 64 * 2;             // one box: BN keys (or 128 rows) x 64 dims bf16
constexpr uint32_t Q_TILE_BYTES = 2 * 128 * 64 * 2;     // 128 rows x 128 dims
constexpr uint32_t BLK_BYTES = 2 * BOX_BYTES;           // one K or V block (BN keys x 128 dims)
// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + Q_TILE_BYTES;
constexpr uint32_t OFF_V = OFF_K + SK * BLK_BYTES;
constexpr uint32_t OFF_BAR = OFF_V + SV * BLK_BYTES;
constexpr uint32_t OFF_STAGE = OFF_K;  // epilogue staging reuses the rings once every MMA has run
// barriers
constexpr int BAR_Q = 0;              // Q tile landed in shared memory
constexpr int BAR_KF = 1;             // [SK] K block landed
constexpr int BAR_KE = BAR_KF + SK;   // [SK] K block consumed by its S product
constexpr int BAR_VF = BAR_KE + SK;   // [SV] V block landed
constexpr int BAR_VE = BAR_VF + SV;   // [SV] V block consumed by its PV product
constexpr int BAR_S = BAR_VE + SV;    // [buf] S ready in TMEM
// p_full is per S/P buffer: softmax may finish block j + 1 before the MMA thread has consumed
// block j, and a single barrier could then complete two phases unobserved.  Block j + 2 cannot
// be written before S(j + 2) is issued, which follows the consumption of block j.
constexpr int BAR_P = BAR_S + 2;      // [buf] P written to TMEM (128 arrivals)
constexpr int BAR_DONE = BAR_P + 2;   // every MMA completed (one-shot)
constexpr int BAR_EPI = BAR_DONE + 1; // staging written (128 arrivals, one-shot)
constexpr int N_BARS = BAR_EPI + 1;
constexpr uint32_t OFF_MISC = OFF_BAR + N_BARS * 8;  // tmem slot, abort flag
constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(128 * 128 * 4 + 128 * 4 <= SK * BLK_BYTES + SV * BLK_BYTES, "staging fits in the rings");
static_assert(BN == 128, "one S/P buffer is 128 columns, P its first 64");

constexpr uint32_t TM_S = 0;    // + buf * 128
constexpr uint32_t TM_O = 256;
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
    const int rb = blockIdx.x % a.nRB;  // 128-row tile within (request, KV head)
    const int kvh = blockIdx.x / a.nRB;
    const int c = blockIdx.y;
    int b = blockIdx.z;  // remapped below to the request this CTA serves

    // Prologue: it overlaps the previous kernel's tail, so it reads nothing it relies on from global
    // memory (the L2 warm-up below only takes a hint from it).
    if (tid == 0) {
        for (int i = 0; i < N_BARS; ++i) {
            uint32_t cnt = 1;
            if (i == BAR_P || i == BAR_P + 1 || i == BAR_EPI) cnt = 128;
            mbar_init(bar(i), cnt);
        }
        *abort_flag = 0;
        fence_mbar_init();
    } else if (tid == 32 * 3) {
        tma_prefetch_desc(&maps.vc);
        tma_prefetch_desc(&maps.vt);
    } else if (tid == 32 * 4) {
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.kc);
        tma_prefetch_desc(&maps.kt);
        if (a.B == 1) {
            // L2 warm-up while the previous kernel finishes: this CTA's Q tile and first K and V
            // blocks, placed by the request's length as it reads now.  A prefetch hands no data to
            // the CTA, and L2 is where every write lands, so a length or cache the previous kernel is
            // still writing costs at most a wasted prefetch; the loads proper follow the wait.
            const int Lh = a.L[0];
            const int k0 = c * chunk_len(a, Lh > 0 && Lh <= a.Lcap ? Lh : 0);
            if (Lh > 0 && Lh <= a.Lcap && k0 < Lh) {
                for (int h = 0; h < 2; ++h) tma_prefetch_l2_3d(&maps.q, h * 64, kvh * a.G, (rb * 128) / a.G);
                const int nbw = min((min(Lh - k0, chunk_len(a, Lh)) + BN - 1) / BN, SK);
                for (int j = 0; j < nbw; ++j)
                    for (int h = 0; h < 2; ++h) {
                        tma_prefetch_l2_4d(&maps.kc, h * 64, kvh, k0 + j * BN, 0);
                        tma_prefetch_l2_4d(&maps.vc, h * 64, kvh, k0 + j * BN, 0);
                    }
            }
        }
    }
    if (warp == 2) {
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
        mark_partial(a, b, kvh, rb, c, -INFINITY);
        if (warp == 2) tmem_dealloc(tmem, 512);
        return;
    }
    if (nck == 1) mark_partial(a, b, kvh, rb, 0, INFINITY);
    const int k0 = c * Cb;
    const int k1 = max(k0, min(Lb, k0 + Cb));
    const int nb_prefix = (k1 - k0 + BN - 1) / BN;
    const bool has_tree = c == tree_chunk;
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
        // ------------------------------------------------------------ TMA producer: Q, then K blocks
        if (lane == 0) {
            const int nz = b * a.Kmax + (rb * 128) / a.G;
            mbar_expect_tx(bar(BAR_Q), Q_TILE_BYTES);
            for (int h = 0; h < 2; ++h)
                tma_load_3d(base + OFF_Q + h * (Q_TILE_BYTES / 2), &maps.q, bar(BAR_Q), h * 64, kvh * a.G, nz);
            for (int j = 0; j < nb; ++j) {
                // a K stage frees as soon as its S product has run
                if (j >= SK && !mbar_wait(bar(BAR_KE + j % SK), ((j / SK) - 1) & 1, wait_ns)) {
                    raise_abort(abort_flag, a.status);
                    break;
                }
                if (aborted(abort_flag)) break;
                load_block(j, &maps.kc, &maps.kt, base + OFF_K + (j % SK) * BLK_BYTES, bar(BAR_KF + j % SK));
                ++k_issued;
            }
        }
    } else if (warp == 3) {
        // ------------------------------------------------------------ TMA producer: V blocks
        if (lane == 0) {
            for (int j = 0; j < nb; ++j) {
                // a V stage frees once its PV product has run
                if (j >= SV && !mbar_wait(bar(BAR_VE + j % SV), ((j / SV) - 1) & 1, wait_ns)) {
                    raise_abort(abort_flag, a.status);
                    break;
                }
                if (aborted(abort_flag)) break;
                load_block(j, &maps.vc, &maps.vt, base + OFF_V + (j % SV) * BLK_BYTES, bar(BAR_VF + j % SV));
                ++v_issued;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (lane 0 alone)
        // tcgen05.mma issue hardly queues ahead of the tensor pipe, so every cycle this thread
        // spends between two products, waits included, is a cycle the pipe idles: one thread runs
        // the loop, and the barrier the next group of products needs is tested (non-blocking) just
        // before the last two products of the current group.
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
            auto kf_of = [&](int j) { return j < nb ? Pre{BAR_KF + j % SK, (uint32_t)((j / SK) & 1)} : none; };
            auto vf_of = [&](int j) { return j < nb ? Pre{BAR_VF + j % SV, (uint32_t)((j / SV) & 1)} : none; };
            // S(j) into S/P buffer j % 2, then the release of K(j)
            auto group_S = [&](int j, Pre nxt) -> bool {
                bool ready = false;
                const uint64_t kd = k_desc + (((j % SK) * BLK_BYTES) >> 4);
                const uint32_t d = tmem + TM_S + (j & 1) * 128;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    if (kk == HD / 16 - 2) ready = test_pre(nxt);
                    const uint32_t off = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
                    mma_bf16_ss(d, q_desc + (off >> 4), kd + (off >> 4), idS, kk > 0);
                }
                mma_commit(bar(BAR_S + (j & 1)));
                mma_commit(bar(BAR_KE + j % SK));
                return ready;
            };
            // O += P(j) V(j), then the release of V(j)
            auto group_PV = [&](int j, Pre nxt) -> bool {
                bool ready = false;
                const uint32_t p = tmem + TM_S + (j & 1) * 128;  // P as packed bf16 pairs
                const uint64_t vd = v_desc + (((j % SV) * BLK_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    if (kk == BN / 16 - 2) ready = test_pre(nxt);
                    mma_bf16_ts(tmem + TM_O, p + kk * 8, vd + ((kk * 2048) >> 4), idO, j > 0 || kk > 0);
                }
                mma_commit(bar(BAR_VE + j % SV));
                return ready;
            };
            bool ok = mbar_wait(bar(BAR_Q), 0, wait_ns) && (nb == 0 || mbar_wait(bar(BAR_KF), 0, wait_ns));
            bool vf_ready = false;
            if (ok && nb > 0) {
                tc_fence_after();
                if (nb > 1) {
                    const bool k1_ready = group_S(0, kf_of(1));
                    ok = wait_pre(kf_of(1), k1_ready);
                    if (ok) {
                        tc_fence_after();
                        vf_ready = group_S(1, vf_of(0));
                    }
                } else {
                    vf_ready = group_S(0, vf_of(0));
                }
            }
            // (the softmax warps zero a ragged block's V rows past the chunk end before they signal
            // P of that block, so its PV, issued after that signal, reads zeros there)
            for (int j = 0; j < nb && ok; ++j) {
                ok = wait_pre(vf_of(j), vf_ready) && mbar_wait(bar(BAR_P + (j & 1)), (j >> 1) & 1, wait_ns) &&
                     !aborted(abort_flag);
                if (!ok) break;
                tc_fence_after();
                if (j + 2 < nb) {
                    const bool kf_ready = group_PV(j, kf_of(j + 2));
                    ok = wait_pre(kf_of(j + 2), kf_ready);
                    if (!ok) break;
                    tc_fence_after();
                    vf_ready = group_S(j + 2, vf_of(j + 1));
                } else {
                    vf_ready = group_PV(j, vf_of(j + 1));
                }
            }
            if (!ok && !aborted(abort_flag)) raise_abort(abort_flag, a.status);
            mma_commit(bar(BAR_DONE));
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax, epilogue
        const int quad = warp & 3;
        const int r = quad * 32 + lane;  // row within the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const int gr = rb * 128 + r;
        const bool row_ok = gr < a.R;
        const int node = row_ok ? gr / a.G : 0;
        const uint64_t anc = row_ok ? a.mask[(size_t)b * a.Kmax + node] : 0ull;
        const float sl2 = a.scale * 1.4426950408889634f;
        float m_used = -INFINITY, l_sum = 0.f;  // running max (log2 units) and row sum
        bool ok = true;
        for (int j = 0; j < nb && ok; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(BAR_S + (j & 1)), (j >> 1) & 1, wait_ns) &&
                                             !aborted(abort_flag));
            if (!ok) break;
            tc_fence_after();
            if (j == ragged_block) {
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
            const uint32_t sbuf = tmem + lane_base + TM_S + (j & 1) * 128;
            float s[BN];
#pragma unroll
            for (int q = 0; q < BN / 32; ++q) tmem_ld32(sbuf + q * 32, s + q * 32);
            tmem_wait_ld();
            const bool tree_blk = j >= nb_prefix;
            if (tree_blk || j == ragged_block) {
                // only the ragged tail and the tree block need masking; tree keys are < 64
                const int valid = tree_blk ? a.Kmax : ragged_valid;
#pragma unroll
                for (int i = 0; i < BN; ++i) {
                    bool keep = i < valid;
                    if (tree_blk) keep = keep && i < 64 && ((anc >> (i & 63)) & 1ull);
                    s[i] = keep ? s[i] : -INFINITY;
                }
            }
            float mx = fmaxf(s[0], s[1]);
#pragma unroll
            for (int i = 2; i < BN; i += 2) mx = fmaxf(mx, fmaxf(s[i], s[i + 1]));
            mx *= sl2;  // sl2 > 0: the maximum commutes with the scale
            if (j == 0) {
                m_used = mx;
            } else if (__any_sync(0xffffffffu, mx > m_used + RESCALE_LOG2)) {
                // raise the running maximum of the rows that need it and rescale their O by
                // 2^(m_used - m_new); the previous PV must have landed first (whole warp).  Its
                // completion is the V-release barrier of block j - 1.  S(j) was committed after
                // PV(j - 2), so that barrier's earlier phase (block j - 1 - SV) has completed, and
                // PV(j - 1 + SV) cannot have completed before this softmax hands over block j: the
                // parity names block j - 1 unambiguously.
                ok = __all_sync(0xffffffffu,
                                mbar_wait(bar(BAR_VE + (j - 1) % SV), ((j - 1) / SV) & 1, wait_ns));
                if (!ok) break;
                tc_fence_after();
                const float m_new = fmaxf(mx, m_used);
                const float alpha = (m_used == -INFINITY) ? 1.f : ex2(m_used - m_new);
                for (int c0 = 0; c0 < HD; c0 += 32) {
                    float o[32];
                    tmem_ld32(tmem + lane_base + TM_O + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= alpha;
                    tmem_st32(tmem + lane_base + TM_O + c0, o);
                }
                tmem_wait_st();
                l_sum *= alpha;
                m_used = m_new;
            }
            const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
            const float2 sc2 = make_float2(sl2, sl2), nm2 = make_float2(neg_m, neg_m);
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float packed[32];
#pragma unroll
                for (int i = 0; i < 64; i += 2) {
                    const float2 x = __ffma2_rn(make_float2(s[hh * 64 + i], s[hh * 64 + i + 1]), sc2, nm2);
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(ex2(x.x), ex2(x.y));
                    // the row sum adds the same rounded weights the PV product uses
                    acc = add_bf16x2_f32(acc, *reinterpret_cast<uint32_t*>(&h2));
                    packed[i / 2] = __uint_as_float(*reinterpret_cast<uint32_t*>(&h2));
                }
                tmem_st32(sbuf + hh * 32, packed);  // P over the first 64 columns of its S buffer
            }
            l_sum += acc.x + acc.y;
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(BAR_P + (j & 1)));
        }
        if (!ok && !aborted(abort_flag)) raise_abort(abort_flag, a.status);
        // ------------------------------------------------------------ epilogue
        if (ok && nb > 0) {
            // every MMA, the last PV included, has completed (one-shot barrier: no phase ambiguity)
            ok = __all_sync(0xffffffffu, mbar_wait(bar(BAR_DONE), 0, wait_ns));
            if (!ok) raise_abort(abort_flag, a.status);
        }
        const bool direct = nck == 1;
        const float inv = (row_ok && l_sum > 0.f) ? 1.f / l_sum : 0.f;
        if (ok) {
            tc_fence_after();
            // stage this thread's row, 16-byte chunks permuted by the row index so a warp's
            // 32 rows spread over all banks
            uint8_t* srow = gbase + OFF_STAGE + r * (direct ? 256 : 512);
            // the row's 128 columns in one round of TMEM loads (the scores' registers are free now)
            float ob[HD];
            if (nb > 0) {
#pragma unroll
                for (int c0 = 0; c0 < HD; c0 += 32) tmem_ld32(tmem + lane_base + TM_O + c0, ob + c0);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < HD; ++i) ob[i] = 0.f;  // no block ran: O was never written
            }
#pragma unroll
            for (int c0 = 0; c0 < HD; c0 += 32) {
                const float* o = ob + c0;
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
        mbar_arrive(bar(BAR_EPI));
        const bool staged = __all_sync(0xffffffffu, mbar_wait(bar(BAR_EPI), 0, wait_ns));
        if (!staged) {
            raise_abort(abort_flag, a.status);
            ok = false;
        }
        if (ok) {
            // write the tile out along contiguous rows; 128 threads
            const uint8_t* stile = gbase + OFF_STAGE;
            if (direct) {
                for (int k = r; k < 128 * 16; k += 128) {
                    const int row = k >> 4, cc = k & 15;
                    const int g = rb * 128 + row;
                    if (g >= a.R) continue;
                    const int nd = g / a.G, hh = kvh * a.G + g % a.G;
                    const uint4 v = *reinterpret_cast<const uint4*>(stile + row * 256 + ((cc ^ (row & 15)) << 4));
                    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.O) +
                                         (((size_t)b * a.Kmax + nd) * a.Hq + hh) * HD + cc * 8;
                    *reinterpret_cast<uint4*>(dst) = v;
                }
            } else {
                const size_t pbase = ((((size_t)b * a.Hkv + kvh) * a.nRB + rb) * a.nchunk + c) * 128;
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
    // ---------------------------------------------------------------- teardown
    if (lane == 0 && (warp == 0 || warp == 3) && aborted(abort_flag)) {
        // loads still in flight write into this CTA's shared memory: each producer waits for
        // the last armed phase of every stage it used (and the Q load) before the CTA may exit
        if (warp == 0) {
            mbar_wait(bar(BAR_Q), 0, kDrainNs);
            for (int st = 0; st < SK; ++st) {
                const int n = (k_issued - st + SK - 1) / SK;
                if (n > 0) mbar_wait(bar(BAR_KF + st), (n - 1) & 1, kDrainNs);
            }
        } else {
            for (int st = 0; st < SV; ++st) {
                const int n = (v_issued - st + SV - 1) / SV;
                if (n > 0) mbar_wait(bar(BAR_VF + st), (n - 1) & 1, kDrainNs);
            }
        }
    }
    if (warp == 2 && lane == 0) {
        // every issued MMA has completed before TMEM is released
        mbar_wait(bar(BAR_DONE), 0, kTeardownNs);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tmem, 512);
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

}  // namespace attn_tc1

int attn_tc1_launch(const AttnArgs& a, cudaStream_t st) {
    using namespace attn_tc1;
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
    dim3 grid(a.nRB * a.Hkv, a.nchunk, a.B);
    launch_pdl(kernel, grid, dim3(NTHREADS), SMEM_BYTES, st, m, a);
    count_launches(1);
    const int rc = launch_status();
    if (rc != GRAFT_OK) return rc;
    return attn_combine_launch(a, st);
}

}  // namespace graft
