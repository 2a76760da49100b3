// Internal layout shared by the host API (mk_api.cu) and the persistent kernel
// (mk_kernel.cu).  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mk.h"

// ---- build-time limits -----------------------------------------------------
#define MK_NCWARPS 8                     // consumer (compute) warps per CTA
#define MK_THREADS ((MK_NCWARPS + 1) * 32) // + one producer (TMA) warp
#define MK_RING 4                        // shared-memory ring slots
#define MK_SLOT 32768                    // bytes per slot: one 256-row x 128-byte TMA box
#define MK_PLANES 1                      // producer lanes issuing copies side by side
#define MK_MAXT 8                        // tokens per verify block (one N=8 MMA tile)
#define MK_MAXKB 32                      // 128-column blocks of the widest GEMV input (4096)
#define MK_MAXE 512                      // routed experts
#define MK_MAXK 8                        // top-k
#define MK_MAXD (MK_MAXT * MK_MAXK)      // distinct experts per layer
#define MK_MAXROWS 64                    // (q heads per kv head) x T
#define MK_MAXSPLIT 160                  // attention splits per kv head
#define MK_ATT_MIN_PAGES 1               // KV pages per attention split, at least
#define MK_MARKS 1024                    // intra-stage trace events per CTA
#define MK_FX 4294967296.0f              // fixed-point scale of the cross-CTA accumulators

#define MK_SCALE_SLOT 2048                // block scales of one tile: FP8 256 x fp32, MXFP4 8 x 256 E8M0

// Dynamic shared memory map (bytes).
#define SM_RING 0
#define SM_SCALE (SM_RING + MK_RING * MK_SLOT)
#define SM_SCRATCH (SM_SCALE + MK_RING * MK_SCALE_SLOT)
#define SM_SCRATCH_BYTES 65536
#define SM_ROUTE (SM_SCRATCH + SM_SCRATCH_BYTES)
#define SM_ROUTE_BYTES 4096
#define SM_BAR (SM_ROUTE + SM_ROUTE_BYTES)
#define SM_MISC (SM_BAR + 256)
#define SM_MISC_BYTES 3072
#define SM_TOTAL (SM_MISC + SM_MISC_BYTES)

// stages of one layer, in stream order
enum { ST_QKV = 0, ST_ATT, ST_O, ST_ROUTER, ST_SHA, ST_EXPA, ST_EXPB, ST_LM };

// one weight matrix, or a stack of E expert matrices, streamed by TMA
struct DMat {
    const CUtensorMap *tmap;   // 64-byte aligned descriptor in device memory
    const float *scale;        // FP8: [E][cols/128][rows]
    const CUtensorMap *smap;   // MXFP4: descriptor of the E8M0 scales [E][cols/32][rows]
    int dtype;                 // MK_DT_*
    int rows, cols;            // per expert
    int n_rg;                  // 256-row groups
    int n_kc;                  // 128-byte column chunks
    int is3d;                  // expert stack
    int es;                    // bytes per stored element (MXFP4: a byte holds two)
    int cpk;                   // columns per 128-byte chunk (MXFP4 256, FP8 128, bf16 64, fp32 32)
    long long scale_estride;   // floats per expert in `scale`
};

struct DLayer {
    const float *attn_norm, *moe_norm, *router_bias;
    DMat qkv, o, router, w1, w3, w2, s1, s3, s2;
};

// control block in device memory.  The barrier counter, which every CTA polls
// at each grid barrier, has a cache line of its own so that the polling does
// not contend with the status words.
struct Ctrl {
    alignas(128) unsigned long long bar_count;  // monotonic grid-barrier arrivals
    alignas(128) int abort;            // set by the first failing wait
    int status;                        // first device error (mk_status)
    int where;                         // diagnostic code of the failing wait
    int pad0;
    unsigned long long epoch;          // bar_count at the start of the next launch
    unsigned long long steps, accepted_sum, distinct_sum;
    int last_accepted, last_distinct;
};

struct DModel {
    int L, H, Hq, Hkv, d, E, K, I, V, P, nshared, max_pages, maxT, G;
    int wdt, rdt, kvdt, kv_es, nqkv;
    float eps;
    long long timeout_ns;
    const DLayer *layers;              // [L]
    const uint16_t *embed;             // bf16 [V][H]
    const float *final_norm;
    DMat lm;
    const float2 *rope;                // [max_pages*P][d/2] (cos, sin)
    // workspace
    Ctrl *ctrl;
    int *att_cnt;                      // [L][Hkv]
    // per-layer accumulators: two copies each, selected by the layer's parity
    long long *qkv_acc;                // [2][MAXT][nqkv]
    long long *res;                    // [MAXT][H]   residual stream
    long long *rlog;                   // [2][MAXT][E]   router logits (un-normalised)
    long long *sh_acc;                 // [2][MAXT][2][I] shared expert gate/up
    long long *ea_acc;                 // [2][MAXT][K][2][I] routed expert gate/up
    long long *logit_acc;              // [MAXT][V]
    float *ssq;                        // [3][MAXKB][MAXT] sum-of-squares partials
    float *o_buf;                      // [MAXT][Hq*d] attention output
    float *att_part;                   // [Hkv][MAXSPLIT][MAXROWS][d+2] attention split partials
    float *cand_v;                     // [G][MAXT] argmax candidates
    int *cand_i;
    float *cand_m, *cand_s;            // [G][MAXT] sampling: slice maximum and sum of exp (log2 domain)
};

struct Params {
    const DModel *m;
    const CUtensorMap *kvmaps;         // [L][2] (K, V)
    void *const *kpool;                // dev array [L]
    void *const *vpool;
    const float *kv_scale;             // dev [L][2]: (K, V) scale of an FP8 E4M3 cache
    const int32_t *page_table;
    const int32_t *tokens;
    const int32_t *positions;
    int T;
    int mode;                          // 0: full step, 1: one layer
    int layer;                         // mode 1
    int n_pages;
    float *out_logits;
    int32_t *out_accepted;
    int32_t *out_argmax;
    float temperature;                 // > 0: verification by sampling (mk_decode_step_sample)
    const float *uniforms;             // sampling: [T] accept tests, then the draw
    int32_t *out_token;                // sampling: the drawn token
    const float *hidden_in;
    float *hidden_out;
    int32_t *out_idx;
    float *out_w;
    int32_t *trace;                    // [L][T][K] routing trace or null
    float *wtrace;                     // [L][T][K] routing weights trace or null
    int host_ctx1;                     // 1 + the ctx the host staged tables for (0: no check)
    unsigned long long *stage_trace;   // [G][cap][2] barrier arrive/release times or null
    int stage_cap;
    unsigned long long *marks;         // [G][MK_MARKS][2] (event id, time) or null
    int skip_barrier;                  // test hook: CTA 0 skips this grid-barrier arrival (0: none)
};

// one kernel per model class (mk_kernel.cu compiled twice): _f32 for all-fp32
// models, _lp for bf16 / FP8 models
cudaError_t mk_launch_f32(const Params &p, int grid, size_t smem, cudaStream_t s);
cudaError_t mk_kernel_setup_f32(size_t smem);
int mk_kernel_max_blocks_f32(size_t smem);
cudaError_t mk_launch_lp(const Params &p, int grid, size_t smem, cudaStream_t s);
cudaError_t mk_kernel_setup_lp(size_t smem);
int mk_kernel_max_blocks_lp(size_t smem);
inline cudaError_t mk_launch(const Params &p, int grid, size_t smem, cudaStream_t s, bool f32) {
    return f32 ? mk_launch_f32(p, grid, smem, s) : mk_launch_lp(p, grid, smem, s);
}
inline cudaError_t mk_kernel_setup(size_t smem, bool f32) {
    return f32 ? mk_kernel_setup_f32(smem) : mk_kernel_setup_lp(smem);
}
inline int mk_kernel_max_blocks(size_t smem, bool f32) {
    return f32 ? mk_kernel_max_blocks_f32(smem) : mk_kernel_max_blocks_lp(smem);
}
