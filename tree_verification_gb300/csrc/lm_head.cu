// Greedy next tokens straight from the target's final hidden states: the
// lm_head product H W^T on the 5th-generation tensor cores with the argmax
// fused into its epilogue, so the [N][V] fp32 logits are never written.
//
// Graft article, architecture paragraph: the merged tree is verified in one
// target forward, and greedy verification needs only the target's argmax at
// each tree node.  g[n] = argmax_v sum_k H[n][k] W[v][k], ties to the lower
// token id.
//
// A persistent CTA per SM computes 128-row x 256-token tiles of logits, each
// over the whole hidden dimension: TMA brings 64-wide k slices of H and W
// (128-byte swizzled boxes) into a 4-stage ring that runs across tiles, one
// lane issues tcgen05.mma (M=128, N=256, K=16, bf16 in, fp32 accumulator in
// TMEM), and four epilogue warps read an accumulator back one row per thread,
// keep the row's first maximum over the tile's tokens and fold it into a
// per-row 64-bit key with atomicMax.  Two accumulators (2 x 256 TMEM
// columns) alternate between tiles, so a tile's epilogue runs while the next
// tile's products do.  The key orders by the logit's value first (its float
// bits mapped to a monotone unsigned order) and then by the complemented
// token id, so the combination is independent of the order tiles finish in
// and ties go to the lower id.  Tiles are numbered row tile fastest and dealt
// round-robin, so the CTAs working at one time cover whole token tiles: each
// W tile is read from HBM once while H stays in L2.
//
// The sampling variant (graft_lm_head_sample) adds Gumbel noise keyed by
// (request, position, token) to every logit / T before the maximum
// (philox.cuh), which draws the target's sample at every node for lossless
// sampling acceptance, again without writing the logits.
//
// Every mbarrier wait is bounded; on timeout the CTA raises
// GRAFT_STATUS_TIMEOUT, drains its loads and releases TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "philox.cuh"
#include "tc_ptx.cuh"

namespace graft {
namespace lmh {

using namespace tc;

constexpr int BM = 128;   // hidden rows per tile
constexpr int BN = 256;   // tokens per tile
constexpr int BK = 64;    // hidden dims per stage (one 128-byte swizzle row)
constexpr int ST = 4;     // ring stages
constexpr int NTHREADS = 192;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = BN * BK * 2;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t OFF_BAR = ST * STAGE_BYTES;
constexpr int BAR_FULL = 0;              // [ST] stage landed
constexpr int BAR_EMPTY = ST;            // [ST] stage consumed by its MMAs
constexpr int BAR_ACC_FULL = 2 * ST;     // [2] an accumulator's tile complete (one phase per use)
constexpr int BAR_ACC_EMPTY = 2 * ST + 2;  // [2] an accumulator read out (128 arrivals per use)
constexpr int BAR_DONE = 2 * ST + 4;     // every MMA completed (one-shot, before TMEM is freed)
constexpr int N_BARS = 2 * ST + 5;
constexpr uint32_t OFF_MISC = OFF_BAR + N_BARS * 8;  // tmem slot, abort flag
constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
constexpr uint64_t kWaitNs = 500000000ull;
constexpr uint64_t kDrainNs = 100000000ull;

struct Maps {
    CUtensorMap h, w;
};

__device__ __forceinline__ uint32_t ordered_bits(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unordered_bits(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

__global__ void __launch_bounds__(256) key_init_kernel(unsigned long long* __restrict__ keys, int N) {
    griddep_enter();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < N; i += gridDim.x * blockDim.x) keys[i] = 0ull;
}

__global__ void __launch_bounds__(256)
key_final_kernel(const unsigned long long* __restrict__ keys, int N, int32_t* __restrict__ argmax,
                 float* __restrict__ max_logit) {
    griddep_enter();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < N; i += gridDim.x * blockDim.x) {
        const unsigned long long k = keys[i];
        argmax[i] = k == 0ull ? 0 : (int32_t)(0xffffffffu - (uint32_t)(k & 0xffffffffull));
        if (max_logit != nullptr) max_logit[i] = k == 0ull ? -INFINITY : unordered_bits((uint32_t)(k >> 32));
    }
}

__device__ __forceinline__ bool aborted(const volatile uint32_t* flag) { return *flag != 0; }
__device__ __forceinline__ void raise_abort(volatile uint32_t* flag, int32_t* status) {
    *flag = 1;
    flag_status(status, GRAFT_STATUS_TIMEOUT);
}

struct SampleArgs {
    const int32_t* tree_pos;  // [N]: node n samples the token at tree_pos[n] + 1
    int Kmax;                 // request of row n = n / Kmax
    float inv_T;
    unsigned long long seed;
};

template <bool SAMPLE>
__global__ void __launch_bounds__(NTHREADS, 1)
lm_head_argmax_kernel(const __grid_constant__ Maps maps, int N, int d, int V, unsigned long long* __restrict__ keys,
                      int32_t* status, SampleArgs sa) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + OFF_MISC);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + OFF_MISC + 4);
    auto bar = [&](int i) { return base + OFF_BAR + 8u * (uint32_t)i; };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nk = (d + BK - 1) / BK;
    const int nrt = (N + BM - 1) / BM;                        // row tiles
    const long long ntiles = (long long)nrt * ((V + BN - 1) / BN);
    // tile t: row tile t % nrt, token tile t / nrt; this CTA takes t = blockIdx.x + i gridDim.x

    if (tid == 0) {
        for (int i = 0; i < N_BARS; ++i)
            mbar_init(bar(i), (i == BAR_ACC_EMPTY || i == BAR_ACC_EMPTY + 1) ? 128 : 1);
        *abort_flag = 0;
        fence_mbar_init();
    } else if (tid == 32) {
        tma_prefetch_desc(&maps.h);
        tma_prefetch_desc(&maps.w);
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

    int issued = 0;
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (lane 0)
        if (lane == 0) {
            int it = 0;  // k slices loaded so far, over every tile of this CTA
            bool ok = true;
            for (long long t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const int row0 = (int)(t % nrt) * BM, v0 = (int)(t / nrt) * BN;
                for (int kt = 0; kt < nk; ++kt, ++it) {
                    const int s = it % ST;
                    if (it >= ST && !mbar_wait(bar(BAR_EMPTY + s), ((it / ST) - 1) & 1, kWaitNs)) {
                        raise_abort(abort_flag, status);
                        ok = false;
                        break;
                    }
                    if (aborted(abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t a = base + s * STAGE_BYTES;
                    mbar_expect_tx(bar(BAR_FULL + s), STAGE_BYTES);
                    tma_load_2d(a, &maps.h, bar(BAR_FULL + s), kt * BK, row0);
                    tma_load_2d(a + A_BYTES, &maps.w, bar(BAR_FULL + s), kt * BK, v0);
                    ++issued;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (lane 0)
        const uint32_t id = idesc_bf16(BM, BN, false, false);
        const uint64_t a_desc = sdesc_sw128(base, 16, 1024);
        const uint64_t b_desc = sdesc_sw128(base + A_BYTES, 16, 1024);
        bool ok = true;
        int it = 0;
        int ti = 0;  // this CTA's tiles so far; tile ti accumulates into buffer ti & 1
        for (long long t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++ti) {
            const int acc = ti & 1;
            if (ti >= 2) {
                // the epilogue has read this buffer's previous tile out
                ok = __all_sync(0xffffffffu, mbar_wait(bar(BAR_ACC_EMPTY + acc), ((ti >> 1) - 1) & 1, kWaitNs) &&
                                                 !aborted(abort_flag));
                if (!ok) break;
                tc_fence_after();
            }
            const uint32_t d_acc = tmem + (uint32_t)acc * BN;
            for (int kt = 0; kt < nk && ok; ++kt, ++it) {
                const int s = it % ST;
                ok = __all_sync(0xffffffffu,
                                mbar_wait(bar(BAR_FULL + s), (it / ST) & 1, kWaitNs) && !aborted(abort_flag));
                if (!ok) break;
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t so = (s * STAGE_BYTES) >> 4;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_bf16_ss(d_acc, a_desc + so + ((kk * 32) >> 4), b_desc + so + ((kk * 32) >> 4), id,
                                    kt > 0 || kk > 0);
                    mma_commit(bar(BAR_EMPTY + s));
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) mma_commit(bar(BAR_ACC_FULL + acc));  // the tile's products complete
            __syncwarp();
        }
        if (!ok && lane == 0 && !aborted(abort_flag)) raise_abort(abort_flag, status);
        if (lane == 0) mma_commit(bar(BAR_DONE));
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue: row argmax (warps 2-5)
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        // the largest Gumbel draw any 32-bit word gives (the draw grows with the word), with a margin
        // for the rounding of its logarithms
        const float g_top = SAMPLE ? gumbel_of(0xffffffffu) + 1e-3f : 0.f;
        int ti = 0;
        for (long long t = blockIdx.x; t < ntiles; t += gridDim.x, ++ti) {
            const int acc = ti & 1;
            const int row0 = (int)(t % nrt) * BM, v0 = (int)(t / nrt) * BN;
            const int n = row0 + r;
            // (the sampler's row loads are issued before the wait for the accumulator, which hides them)
            uint32_t nb = 0, npos = 0;
            unsigned long long key_seen = 0ull;
            if (SAMPLE && n < N) {
                nb = (uint32_t)(n / sa.Kmax);
                npos = (uint32_t)(sa.tree_pos[n] + 1);
                // the row's key as other tiles have raised it so far (any value read is a real score)
                key_seen = __ldcg(keys + n);
            }
            const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(BAR_ACC_FULL + acc), (ti >> 1) & 1, kWaitNs)) &&
                            !aborted(abort_flag);
            if (!ok) {
                if (!aborted(abort_flag)) raise_abort(abort_flag, status);
                break;
            }
            tc_fence_after();
            float best = -INFINITY;
            int bi = -1;
            // a score another tile reached in this row, if any (sampling); until a row of the warp has
            // one, the warp draws every token's noise without the tests below
            const float reached = key_seen != 0ull ? unordered_bits((uint32_t)(key_seen >> 32)) : -INFINITY;
            const bool prune = SAMPLE && __any_sync(0xffffffffu, key_seen != 0ull);

            for (int c0 = 0; c0 < BN; c0 += 32) {
                float x[32];
                tmem_ld32(tmem + (uint32_t)acc * BN + ((uint32_t)(quad * 32) << 16) + c0, x);
                tmem_wait_ld();
                if (c0 == BN - 32) {
                    // the accumulator is in registers: the tile after next may overwrite it
                    tc_fence_before();
                    mbar_arrive(bar(BAR_ACC_EMPTY + acc));
                }
                if (SAMPLE && !prune) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const uint4 r4 = noise_draws(sa.seed, nb, npos, (uint32_t)((v0 + c0 + i) >> 2));
                        x[i] = x[i] * sa.inv_T + gumbel_of(r4.x);
                        x[i + 1] = x[i + 1] * sa.inv_T + gumbel_of(r4.y);
                        x[i + 2] = x[i + 2] * sa.inv_T + gumbel_of(r4.z);
                        x[i + 3] = x[i + 3] * sa.inv_T + gumbel_of(r4.w);
                    }
                } else if (SAMPLE) {
                    // A token whose scaled logit plus the largest draw (g_top) stays below a score
                    // already reached in its row cannot be the row's pick: four such tokens draw no
                    // noise and score -inf.  The bound allows for the rounding of the sums (a relative
                    // 2^-20).
                    const float top = fmaxf(reached, best);
                    const float lim = top - g_top - fabsf(top) * 9.5367431640625e-7f;
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float s0 = x[i] * sa.inv_T, s1 = x[i + 1] * sa.inv_T;
                        const float s2 = x[i + 2] * sa.inv_T, s3 = x[i + 3] * sa.inv_T;
                        if (fmaxf(fmaxf(s0, s1), fmaxf(s2, s3)) >= lim) {
                            const uint4 r4 = noise_draws(sa.seed, nb, npos, (uint32_t)((v0 + c0 + i) >> 2));
                            x[i] = s0 + gumbel_of(r4.x);
                            x[i + 1] = s1 + gumbel_of(r4.y);
                            x[i + 2] = s2 + gumbel_of(r4.z);
                            x[i + 3] = s3 + gumbel_of(r4.w);
                        } else {
                            x[i] = x[i + 1] = x[i + 2] = x[i + 3] = -INFINITY;
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int v = v0 + c0 + i;
                    if (v < V && x[i] > best) {  // ascending ids, strict: the first maximum stays
                        best = x[i];
                        bi = v;
                    }
                }
            }
            if (n < N && bi >= 0) {
                const unsigned long long key = ((unsigned long long)ordered_bits(best) << 32) |
                                               (unsigned long long)(0xffffffffu - (uint32_t)bi);
                atomicMax(keys + n, key);
            }
        }
    }
    // ---------------------------------------------------------------- teardown
    if (warp == 0 && lane == 0 && aborted(abort_flag)) {
        for (int s = 0; s < ST; ++s) {
            const int uses = (issued - s + ST - 1) / ST;
            if (uses > 0) mbar_wait(bar(BAR_FULL + s), (uses - 1) & 1, kDrainNs);
        }
    }
    if (warp == 1 && lane == 0) mbar_wait(bar(BAR_DONE), 0, kWaitNs);
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

bool encode_rows(CUtensorMap* m, const void* ptr, int rows, int d, int box_rows) {
    auto enc = encoder();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    cuuint32_t box[2] = {BK, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace lmh
}  // namespace graft

using namespace graft;

extern "C" int graft_lm_head_argmax_workspace_size(int N, size_t* bytes) {
    if (bytes == nullptr || N < 0) return GRAFT_ERR_INVALID_ARG;
    WsCarver c(nullptr);
    c.take<unsigned long long>((size_t)N);
    *bytes = c.bytes();
    return GRAFT_OK;
}

namespace {

int lm_head_impl(int N, int d_model, int V, const void* H, const void* W_lm, int32_t* argmax, float* max_logit,
                 const lmh::SampleArgs* sa, int32_t* status, void* ws, size_t ws_bytes, graft_stream_t stream) {
    using namespace lmh;
    if (N < 0 || d_model < 1 || V < 1) return GRAFT_ERR_INVALID_ARG;
    if (N == 0) return GRAFT_OK;
    if (H == nullptr || W_lm == nullptr || argmax == nullptr) return GRAFT_ERR_INVALID_ARG;
    if ((d_model % 8) != 0) return GRAFT_ERR_UNSUPPORTED_SHAPE;  // 16-byte row pitch for TMA
    if (((reinterpret_cast<uintptr_t>(H) | reinterpret_cast<uintptr_t>(W_lm)) & 15) != 0) return GRAFT_ERR_INVALID_ARG;
    const long long row_tiles = ((long long)N + BM - 1) / BM, tok_tiles = ((long long)V + BN - 1) / BN;
    if (row_tiles > (1LL << 31) - 1 || tok_tiles > 65535) return GRAFT_ERR_UNSUPPORTED_SHAPE;
    WsCarver sizer(nullptr);
    sizer.take<unsigned long long>((size_t)N);
    if (!ws_ok(ws, ws_bytes, sizer.bytes())) return GRAFT_ERR_WORKSPACE;
    WsCarver c(ws);
    unsigned long long* keys = c.take<unsigned long long>((size_t)N);
    Maps m;
    if (!encode_rows(&m.h, H, N, d_model, BM) || !encode_rows(&m.w, W_lm, V, d_model, BN)) return GRAFT_ERR_CUDA;
    static bool attr_set[2][64] = {{false}};
    const int smp = sa != nullptr;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[smp][dev]) {
        const cudaError_t e =
            smp ? cudaFuncSetAttribute(lm_head_argmax_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES)
                : cudaFuncSetAttribute(lm_head_argmax_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
        if (!cuda_ok(e)) return GRAFT_ERR_CUDA;
        attr_set[smp][dev] = true;
    }
    cudaStream_t st = (cudaStream_t)stream;
    const unsigned small = (unsigned)((N + 255) / 256 < 1024 ? (N + 255) / 256 : 1024);
    // persistent: one CTA per SM (shared memory allows no more), at most one per tile
    const long long tiles = row_tiles * tok_tiles;
    int sms = device_sm_count();
    if (sms <= 0) sms = 148;
    const dim3 grid((unsigned)(tiles < sms ? tiles : sms));
    launch_pdl(key_init_kernel, dim3(small), dim3(256), 0, st, keys, N);
    if (smp)
        launch_pdl(lm_head_argmax_kernel<true>, grid, dim3(NTHREADS), SMEM_BYTES, st, m, N, d_model, V, keys, status,
                   *sa);
    else
        launch_pdl(lm_head_argmax_kernel<false>, grid, dim3(NTHREADS), SMEM_BYTES, st, m, N, d_model, V, keys, status,
                   SampleArgs{nullptr, 1, 1.f, 0ull});
    launch_pdl(key_final_kernel, dim3(small), dim3(256), 0, st, keys, N, argmax, max_logit);
    count_launches(3);
    return launch_status();
}

}  // namespace

extern "C" int graft_lm_head_argmax(int N, int d_model, int V, const void* H, const void* W_lm, int32_t* argmax,
                                    float* max_logit, int32_t* status, void* ws, size_t ws_bytes,
                                    graft_stream_t stream) {
    return lm_head_impl(N, d_model, V, H, W_lm, argmax, max_logit, nullptr, status, ws, ws_bytes, stream);
}

extern "C" int graft_lm_head_sample(int N, int d_model, int V, const void* H, const void* W_lm, int Kmax,
                                    const int32_t* tree_pos, float temperature, uint64_t seed, int32_t* sampled,
                                    int32_t* status, void* ws, size_t ws_bytes, graft_stream_t stream) {
    if (Kmax < 1 || tree_pos == nullptr || !(temperature > 0.f) || (N > 0 && N % Kmax != 0))
        return GRAFT_ERR_INVALID_ARG;
    const lmh::SampleArgs sa{tree_pos, Kmax, 1.0f / temperature, (unsigned long long)seed};
    return lm_head_impl(N, d_model, V, H, W_lm, sampled, nullptr, &sa, status, ws, ws_bytes, stream);
}
