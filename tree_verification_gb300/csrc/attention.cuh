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
    int cluster;                  // one-tile kernel: chunks reduced in a thread-block cluster (0: off)
    int C;                        // prefix keys per chunk (multiple of 128)
    int nchunk;                   // chunks per (request, KV head) allowed by Lcap
    int Lcap;
    float scale;
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
};

// Warp-level mma.sync path: any group size; 128-row CTAs.
int attn_mma_launch(const AttnArgs& a, cudaStream_t st);
// tcgen05 path: group sizes dividing 128; CTAs of two 128-row tiles
// (attn_tc_launch) or of one (attn_tc1_launch), as a.tiles says.
bool attn_tc_supported(int G);
int attn_tc_launch(const AttnArgs& a, cudaStream_t st);
int attn_tc1_launch(const AttnArgs& a, cudaStream_t st);
// Merges split-key partials (no-op when every request fits one chunk or a
// cluster reduced them).
int attn_combine_launch(const AttnArgs& a, cudaStream_t st);

}  // namespace graft
