// Tree-masked GQA attention, warp-level mma.sync path (bf16 in, fp32 accumulate).
//
// Graft article, architecture paragraph: the hybrid tree is verified on the
// standard tree-attention path in one target forward; Graft abstract: large
// trees cost VRAM bandwidth and compute.  For request b, KV head g and tree
// node i, every query head h of g's group attends to all L[b] prefix keys of
// the cache plus the tree keys in node i's ancestor-or-self mask.
//
// Decomposition: one CTA per (request, KV head, 128-row block of the
// Kmax * group query rows, key chunk).  Keys are split into chunks so that
// small batches still fill the GPU; the last chunk of a request also takes
// the tree block (Kmax <= 64 keys, masked by the ancestor bits).  A request
// that fits one chunk writes O directly; otherwise each chunk writes a
// normalised fp32 partial with its log2-sum-exp and attn_combine_kernel
// merges them.  K/V tiles of 64 keys are double-buffered in shared memory
// with cp.async; QK^T and PV run on mma.sync.m16n8k16.
#include <cmath>

#include "attention.cuh"
#include "common.cuh"

namespace graft {
namespace attn_mma {

constexpr int HD = GRAFT_HEAD_DIM;
constexpr int BM = 128;
constexpr int BN = 64;
constexpr int NT = 256;
constexpr int TILE_BYTES = BN * HD * 2;
constexpr int SMEM = BM * HD * 2 + 4 * TILE_BYTES;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// byte offset of 16-byte chunk ch (0..15) of row r in a [rows][128] bf16 tile
__device__ __forceinline__ uint32_t swz(int r, int ch) {
    return (uint32_t)(r * (HD * 2) + ((ch ^ (r & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(NT)
attn_partial_kernel(AttnArgs a) {
    griddep_enter();
    extern __shared__ __align__(128) unsigned char smem[];
    const int nRB = a.nRB;
    const int rb = blockIdx.x % nRB;
    const int kvh = blockIdx.x / nRB;
    const int c = blockIdx.y;
    const int b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const int Lb = a.L[b];
    if (Lb < 0 || Lb > a.Lcap) {
        if (c == 0 && tid == 0 && rb == 0 && kvh == 0) flag_status(a.status, GRAFT_STATUS_LENGTH);
        mark_partial(a, b, kvh, rb, c, -INFINITY);
        return;
    }
    const int Cb = chunk_len(a, Lb);
    const int nck = Lb > 0 ? (Lb + Cb - 1) / Cb : 1;
    if (c >= nck) {
        mark_partial(a, b, kvh, rb, c, -INFINITY);
        return;
    }
    if (nck == 1) mark_partial(a, b, kvh, rb, 0, INFINITY);
    const int k0 = c * Cb;
    const int k1 = min(Lb, k0 + Cb);
    const int nb_prefix = (k1 - k0 + BN - 1) / BN;
    const bool has_tree = (c == nck - 1);
    const int nb = nb_prefix + (has_tree ? 1 : 0);

    const uint32_t sQ = smem_u32(smem);
    const uint32_t sK = sQ + BM * HD * 2;
    const uint32_t sV = sK + 2 * TILE_BYTES;

    const __nv_bfloat16* Q = reinterpret_cast<const __nv_bfloat16*>(a.Q);
    const __nv_bfloat16* Kc = reinterpret_cast<const __nv_bfloat16*>(a.Kc);
    const __nv_bfloat16* Vc = reinterpret_cast<const __nv_bfloat16*>(a.Vc);
    const __nv_bfloat16* Kt = reinterpret_cast<const __nv_bfloat16*>(a.Kt);
    const __nv_bfloat16* Vt = reinterpret_cast<const __nv_bfloat16*>(a.Vt);

    // Q tile: row r -> global row rb*128 + r -> (node, head)
    for (int i = tid; i < BM * 16; i += NT) {
        const int r = i >> 4, ch = i & 15;
        const int gr = rb * BM + r;
        const bool v = gr < a.R;
        const int node = v ? gr / a.G : 0;
        const int h = kvh * a.G + (v ? gr % a.G : 0);
        const __nv_bfloat16* src = Q + (((size_t)b * a.Kmax + node) * a.Hq + h) * HD + ch * 8;
        cp_async16(sQ + swz(r, ch), src, v);
    }
    auto load_block = [&](int bi, int buf) {
        const uint32_t dK = sK + buf * TILE_BYTES, dV = sV + buf * TILE_BYTES;
        if (bi < nb_prefix) {
            const int start = k0 + bi * BN;
            for (int i = tid; i < BN * 16; i += NT) {
                const int r = i >> 4, ch = i & 15;
                const int key = start + r;
                const bool v = key < k1;
                const size_t off = (((size_t)b * a.Lcap + (v ? key : 0)) * a.Hkv + kvh) * HD + ch * 8;
                cp_async16(dK + swz(r, ch), Kc + off, v);
                cp_async16(dV + swz(r, ch), Vc + off, v);
            }
        } else {
            for (int i = tid; i < BN * 16; i += NT) {
                const int r = i >> 4, ch = i & 15;
                const bool v = r < a.Kmax;
                const size_t off = (((size_t)b * a.Kmax + (v ? r : 0)) * a.Hkv + kvh) * HD + ch * 8;
                cp_async16(dK + swz(r, ch), Kt + off, v);
                cp_async16(dV + swz(r, ch), Vt + off, v);
            }
        }
    };
    load_block(0, 0);
    cp_commit();

    // ancestor masks of this thread's two rows (g = lane/4 and g + 8 within the warp's 16)
    uint64_t anc[2];
    bool row_ok[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        const int gr = rb * BM + warp * 16 + (lane >> 2) + h2 * 8;
        row_ok[h2] = gr < a.R;
        anc[h2] = row_ok[h2] ? a.mask[(size_t)b * a.Kmax + gr / a.G] : 0ull;
    }

    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    uint32_t qf[8][4];
    const float sl2 = a.scale * 1.4426950408889634f;

    for (int bi = 0; bi < nb; ++bi) {
        if (bi + 1 < nb) load_block(bi + 1, (bi + 1) & 1);
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        if (bi == 0) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int r = warp * 16 + (lane & 15);
                const int ch = kk * 2 + (lane >> 4);
                ldsm_x4(sQ + swz(r, ch), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
            }
        }
        const uint32_t tK = sK + (bi & 1) * TILE_BYTES, tV = sV + (bi & 1) * TILE_BYTES;
        float s[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                const int m = lane >> 3;
                const int key = np * 16 + (m >> 1) * 8 + (lane & 7);
                const int ch = kk * 2 + (m & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(tK + swz(key, ch), b0, b1, b2, b3);
                mma16816(s[2 * np], qf[kk], b0, b1);
                mma16816(s[2 * np + 1], qf[kk], b2, b3);
            }
        }
        // mask, scale into the log2 domain, online softmax
        const bool tree_blk = bi >= nb_prefix;
        const int valid = tree_blk ? a.Kmax : min(BN, k1 - (k0 + bi * BN));
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = nt * 8 + (lane & 3) * 2 + (e & 1);
                const int h2 = e >> 1;
                bool ok = col < valid;
                if (tree_blk) ok = ok && ((anc[h2] >> col) & 1ull);
                const float v = ok ? s[nt][e] * sl2 : -INFINITY;
                s[nt][e] = v;
                mx[h2] = fmaxf(mx[h2], v);
            }
        }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 1));
            mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 2));
        }
        float base[2], alpha[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const float mn = fmaxf(m_run[h2], mx[h2]);
            base[h2] = (mn == -INFINITY) ? 0.f : mn;
            alpha[h2] = fast_exp2(m_run[h2] - base[h2]);
            m_run[h2] = mn;
        }
        float rs[2] = {0.f, 0.f};
        uint32_t pa[4][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            float p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) p[e] = fast_exp2(s[nt][e] - base[e >> 1]);
            // the row sum uses the bf16-rounded weights that the PV product consumes
            const __nv_bfloat162 w01 = __floats2bfloat162_rn(p[0], p[1]);
            const __nv_bfloat162 w23 = __floats2bfloat162_rn(p[2], p[3]);
            rs[0] += __low2float(w01) + __high2float(w01);
            rs[1] += __low2float(w23) + __high2float(w23);
            const int ks = nt >> 1;
            if ((nt & 1) == 0) {
                pa[ks][0] = *reinterpret_cast<const uint32_t*>(&w01);
                pa[ks][1] = *reinterpret_cast<const uint32_t*>(&w23);
            } else {
                pa[ks][2] = *reinterpret_cast<const uint32_t*>(&w01);
                pa[ks][3] = *reinterpret_cast<const uint32_t*>(&w23);
            }
        }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) l_run[h2] = l_run[h2] * alpha[h2] + rs[h2];
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) {
            o[dt][0] *= alpha[0];
            o[dt][1] *= alpha[0];
            o[dt][2] *= alpha[1];
            o[dt][3] *= alpha[1];
        }
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int dp = 0; dp < 8; ++dp) {
                const int m = lane >> 3;
                const int key = ks * 16 + (m & 1) * 8 + (lane & 7);
                const int ch = dp * 2 + (m >> 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(tV + swz(key, ch), b0, b1, b2, b3);
                mma16816(o[2 * dp], pa[ks], b0, b1);
                mma16816(o[2 * dp + 1], pa[ks], b2, b3);
            }
        }
        __syncthreads();
    }
    cp_wait<0>();

#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        l_run[h2] += __shfl_xor_sync(0xffffffffu, l_run[h2], 1);
        l_run[h2] += __shfl_xor_sync(0xffffffffu, l_run[h2], 2);
    }
    const bool direct = (nck == 1);
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        if (!row_ok[h2]) continue;
        const int r = warp * 16 + (lane >> 2) + h2 * 8;
        const int gr = rb * BM + r;
        const float inv = 1.f / l_run[h2];
        if (direct) {
            const int node = gr / a.G, h = kvh * a.G + gr % a.G;
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.O) + (((size_t)b * a.Kmax + node) * a.Hq + h) * HD;
#pragma unroll
            for (int dt = 0; dt < 16; ++dt) {
                const int col = dt * 8 + (lane & 3) * 2;
                *reinterpret_cast<__nv_bfloat162*>(dst + col) =
                    __floats2bfloat162_rn(o[dt][2 * h2] * inv, o[dt][2 * h2 + 1] * inv);
            }
        } else {
            const size_t pi = ((((size_t)b * a.Hkv + kvh) * nRB + rb) * a.nchunk + c) * BM + r;
            float* dst = a.part_o + pi * HD;
#pragma unroll
            for (int dt = 0; dt < 16; ++dt) {
                const int col = dt * 8 + (lane & 3) * 2;
                *reinterpret_cast<float2*>(dst + col) = make_float2(o[dt][2 * h2] * inv, o[dt][2 * h2 + 1] * inv);
            }
            if ((lane & 3) == 0) a.part_lse[pi] = m_run[h2] + log2f(l_run[h2]);
        }
    }
}

}  // namespace attn_mma

// Merges the per-chunk partial outputs of every (request, KV head, row) in
// one pass: O = sum_c 2^(lse_c - lse) O_c with lse = log2 sum_c 2^lse_c,
// kept as a running maximum.  The attention kernels mark chunks past a
// request's keys with lse = -inf and rows already written directly with
// lse_0 = +inf, so the merge needs no request length.  One warp per output
// row, four dims per lane; the loads of up to kMergeBatch chunks are issued
// together, so a row costs one memory round trip per kMergeBatch chunks: 16,
// or 20 when a call has more chunks (the 19 of a 65536-token prefix over 152
// SMs then take one round trip, where the unused slots of a wider batch would
// cost the calls with few chunks more than they save).
template <int kMergeBatch>
__global__ void __launch_bounds__(256, 2)
attn_combine_kernel(AttnArgs a) {
    griddep_enter();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 8 + warp;
    const long long total = (long long)a.B * a.Hkv * a.nRB * 128;
    if (row >= total) return;
    const int r = (int)(row % 128);
    const int tile = (int)((row / 128) % a.nRB);
    const int kvh = (int)((row / (128LL * a.nRB)) % a.Hkv);
    const int b = (int)(row / (128LL * a.nRB * a.Hkv));
    const int gr = tile * 128 + r;
    if (gr >= a.R) return;
    const size_t base = (((size_t)b * a.Hkv + kvh) * a.nRB + tile) * a.nchunk;
    const float* lse = a.part_lse + base * 128 + r;
    const float* po = a.part_o + (base * 128 + r) * GRAFT_HEAD_DIM + lane * 4;
    float m = -INFINITY, l = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < a.nchunk; c0 += kMergeBatch) {
        float lc[kMergeBatch];
        float4 v[kMergeBatch];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
            const int c = c0 + u;
            lc[u] = c < a.nchunk ? lse[(size_t)c * 128] : -INFINITY;
            v[u] = c < a.nchunk ? *reinterpret_cast<const float4*>(po + (size_t)c * 128 * GRAFT_HEAD_DIM)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (c0 == 0 && lc[0] == INFINITY) return;  // written directly by the attention kernel
        float mb = m;
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) mb = fmaxf(mb, lc[u]);
        if (mb == -INFINITY) continue;  // nothing from this batch (uniform over the warp)
        if (mb > m) {
            const float s = (m == -INFINITY) ? 0.f : exp2f(m - mb);
            acc.x *= s;
            acc.y *= s;
            acc.z *= s;
            acc.w *= s;
            l *= s;
            m = mb;
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
            if (lc[u] == -INFINITY) continue;  // chunk past the request's keys: its loaded partial is garbage
            const float w = exp2f(lc[u] - m);
            acc.x += w * v[u].x;
            acc.y += w * v[u].y;
            acc.z += w * v[u].z;
            acc.w += w * v[u].w;
            l += w;
        }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int node = gr / a.G, h = kvh * a.G + gr % a.G;
    __nv_bfloat16* dst =
        reinterpret_cast<__nv_bfloat16*>(a.O) + (((size_t)b * a.Kmax + node) * a.Hq + h) * GRAFT_HEAD_DIM + lane * 4;
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 v;
    v.x = *reinterpret_cast<uint32_t*>(&lo);
    v.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst) = v;
}

int attn_combine_launch(const AttnArgs& a, cudaStream_t st) {
    if (a.nchunk <= 1) return GRAFT_OK;
    const long long rows = (long long)a.B * a.Hkv * a.nRB * 128;
    const dim3 grid((unsigned)((rows + 7) / 8));
    if (a.nchunk > 16)
        launch_pdl(attn_combine_kernel<20>, grid, dim3(256), 0, st, a);
    else
        launch_pdl(attn_combine_kernel<16>, grid, dim3(256), 0, st, a);
    count_launches(1);
    return launch_status();
}

namespace attn_mma {
}  // namespace attn_mma

int attn_mma_launch(const AttnArgs& a, cudaStream_t st) {
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        if (!cuda_ok(cudaFuncSetAttribute(attn_mma::attn_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 attn_mma::SMEM)))
            return GRAFT_ERR_CUDA;
        attr_set[dev] = true;
    }
    dim3 grid(a.nRB * a.Hkv, a.nchunk, a.B);
    launch_pdl(attn_mma::attn_partial_kernel, dim3(grid), dim3(attn_mma::NT), attn_mma::SMEM, st, a);
    count_launches(1);
    const int rc = launch_status();
    if (rc != GRAFT_OK) return rc;
    return attn_combine_launch(a, st);
}

}  // namespace graft
