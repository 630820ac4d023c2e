// Arguments shared by the tree-attention kernels and their host dispatch.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace graft {

// Keys per block of the tcgen05 path; key chunks are multiples of it.
constexpr int ATTN_TC_BLOCK_KEYS = 128;

struct AttnArgs {
    int B, Hq, Hkv, G, Kmax, R;  // R = Kmax * G query rows per (request, KV head)
    int nRB;                      // 128-row blocks per (request, KV head)
    int tiles;                    // tcgen05 path: 128-row tiles per CTA (1 or 2)
    int C;                        // minimum prefix keys per chunk (multiple of 128)
    int nchunk;                   // chunk CTAs per (request, KV head, row tile)
    int Lcap;
    float scale;
    uint64_t wait_ns;  // bound on every pipeline wait inside the kernels (0.5 s unless tuned)
    const void* Q;
    const void* Kc;
    const void* Vc;
    const void* Kt;
    const void* Vt;
    const int32_t* L;
    const uint64_t* mask;
    void* O;
    float* part_o;    // [B][Hkv][nRB][nchunk][128][128] normalised partial outputs
    float* part_lse;  // [B][Hkv][nRB][nchunk][128] log2-sum-exp of each partial
    int32_t* status;
    // stream schedule (attention_tcs.cu): items cut at a CTA-group boundary
    int32_t* cut_cnt;  // [items][2] arrival counters (zero between calls)
    float* cut_o;      // [2 ctas][2][32][128] float4: partial rows of the cut pieces, chunk-major
                       // (float4 column chunk x of the 128 rows side by side; two slots per CTA)
    float* cut_lse;    // [2 ctas][2][128] their log2-sum-exp
};

// Marks the log2-sum-exp slots of one 128-row tile's partial for chunk c:
// -inf for a chunk past the request's keys (it contributes nothing), +inf
// for chunk 0 of a request that fits one chunk (its output was written
// directly, so the merge leaves the rows alone).  No-op without partials.
static __device__ __noinline__ void mark_partial(const AttnArgs& a, int b, int kvh, int tile, int c, float value) {
    if (a.nchunk <= 1 || a.part_lse == nullptr || tile >= a.nRB) return;
    const size_t base = ((((size_t)b * a.Hkv + kvh) * a.nRB + tile) * a.nchunk + c) * 128;
    for (int r = threadIdx.x; r < 128; r += blockDim.x) a.part_lse[base + r] = value;
}

// Prefix keys per chunk for a request of Lb keys: its keys split evenly over
// the a.nchunk chunk CTAs in whole 128-key blocks, never fewer than a.C.  The
// split follows each request's own length, not the cache capacity, so a cache
// sized far beyond the current prefixes still spreads them over the SMs.
// Chunks past ceil(Lb / chunk) hold no prefix keys.
static __device__ __forceinline__ int chunk_len(const AttnArgs& a, int Lb) {
    const int per = (Lb + a.nchunk - 1) / a.nchunk;
    const int blk = (per + ATTN_TC_BLOCK_KEYS - 1) / ATTN_TC_BLOCK_KEYS * ATTN_TC_BLOCK_KEYS;
    return blk > a.C ? blk : a.C;
}
// Warp-level mma.sync path: any group size; 128-row CTAs.
int attn_mma_launch(const AttnArgs& a, cudaStream_t st);
// tcgen05 path: group sizes dividing 128; CTAs of two 128-row tiles
// (attn_tc_launch) or of one (attn_tc1_launch), as a.tiles says.
bool attn_tc_supported(int G);
int attn_tc_launch(const AttnArgs& a, cudaStream_t st);
int attn_tc1_launch(const AttnArgs& a, cudaStream_t st);
// Persistent two-tile kernel (attention_tcp.cu): the work items of the two-tile grid (nRB even)
// dealt to `ctas` CTAs that run theirs back to back; then the merge, as attn_tc_launch.
int attn_tcp_items(const AttnArgs& a);
int attn_tcp_launch(const AttnArgs& a, int ctas, cudaStream_t st);
// Persistent two-tile kernel with the stream schedule (attention_tcs.cu): one key chunk per request,
// B <= 256, `ctas` a multiple of nRB / 2; the key blocks split evenly over the CTAs, cut items merged
// by their last piece through the arrival counters a.cut_cnt.
int attn_tcs_launch(const AttnArgs& a, int ctas, cudaStream_t st);
// Merges split-key partials (no-op when every request fits one chunk).
int attn_combine_launch(const AttnArgs& a, cudaStream_t st);

}  // namespace graft
