// Persistent verify-step megakernel for sm_103a.
//
// One cooperative launch runs a whole speculative-verify step: embedding, every
// decoder layer (RMSNorm + QKV GEMV + RoPE + KV append + split-K GQA attention,
// O projection + residual, router GEMV + sigmoid + bitonic top-k, routed and
// shared SwiGLU experts + residual), the final norm, the LM head, argmax and the
// accept-prefix count.  This replaces the ~1,300 small kernels per step that the
// single-GB300 decode analysis ("Why one GB300 doesn't beat 4x RTX PRO 6000 at
// single-stream decode", section "Where the 11.2 ms goes") counts, and keeps one
// persistent CTA per SM as the megakernel plugin does ("DeepSeek-V4.1-Flash breaks
// 1,000 tokens per second for one user", section "What NVIDIA shipped").
//
// Structure of a CTA (288 threads, one CTA per SM):
//   warp 8      producer: walks the CTA's static tile schedule for the whole
//               step and streams weight tiles (256 rows x 128 bytes, one TMA box
//               with the 128-byte swizzle) and KV pages into a 4-slot shared
//               memory ring with cp.async.bulk.tensor, plus 1-D bulk copies of
//               the FP8 block scales, all with an L2 evict-first hint.  It runs
//               ahead across grid barriers; it only stops for a free slot, and
//               for the router result before the routed-expert tiles of a layer.
//   warps 0..7  consumers: warp w reduces rows 32w..32w+31 of each tile against
//               the T <= 8 activations with mma.sync m16n8k16 (tokens are the
//               N = 8 side; FP8 codes are widened to f16 in registers and the
//               1x128 scales applied per block), accumulating across consecutive
//               tiles of an item, then adds its partial into a global fixed-point
//               (2^-32) int64 accumulator.  Integer adds make every cross-CTA
//               reduction order-independent, so the step is bitwise deterministic.
// RMSNorm is folded: GEMVs consume gamma*x and the consumer of their result
// divides by rms(x); the per-block sums of squares are formed while the
// activation fragments are built.  Grid barriers separate the stages: one
// release reduction per CTA on a monotonic counter, acquire polls to wait.
// Every wait is bounded by %globaltimer and turns into a status code.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math_constants.h>

#include "mk_internal.h"

// This file is compiled twice: with MK_F32_MODEL=1 for all-fp32 models (FFMA
// GEMV tiles, FFMA attention over head_dim 64) and with MK_F32_MODEL=0 for
// bf16 / FP8 models (tensor-core tiles and attention).  Each kernel then holds
// only the code paths its models take, which keeps it small for the
// instruction cache: most of the step's code runs once per layer.
#ifndef MK_F32_MODEL
#define MK_F32_MODEL 0
#endif

namespace {

constexpr bool kF32 = MK_F32_MODEL != 0;

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t sa(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t tx) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sa(b)), "r"(tx)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(sa(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// TMA tile and bulk copies into shared memory, completing on an mbarrier, with
// an L2 eviction-priority hint (streamed weights are read once per step: evict
// them first so that activations, accumulators, tensor maps and code stay
// resident in L2)
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma2d_h(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                        uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(sa(dst)),
        "l"(map), "r"(x), "r"(y), "r"(sa(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma3d_h(void *dst, const CUtensorMap *map, int x, int y, int z,
                                        uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(sa(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(sa(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void bulk_g2s_h(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                           uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(sa(dst)),
        "l"(src), "r"(bytes), "r"(sa(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void bar_consumers() {
    asm volatile("bar.sync 1, %0;" ::"n"(MK_NCWARPS * 32) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void ldsm4(uint32_t a, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                      uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(a));
}
__device__ __forceinline__ void ldsm4t(uint32_t a, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                       uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(a));
}
__device__ __forceinline__ void mma_f16(float *c, uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float *c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// four FP8 E4M3 codes (byte 0 first) -> two f16x2 words (bytes 0,1 and 2,3)
__device__ __forceinline__ void e4m3x4_f16(uint32_t v, uint32_t &lo, uint32_t &hi) {
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.rn.f16x2.e4m3x2 %0, l;\n"
        " cvt.rn.f16x2.e4m3x2 %1, h;\n}\n"
        : "=r"(lo), "=r"(hi)
        : "r"(v));
}
// FP8 E4M3 code of x: nearest, ties to even, saturating at +-448
__device__ __forceinline__ unsigned char e4m3_code(float x) {
    return (unsigned char)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}
// bytes of a and b picked by selector sel (prmt: a's bytes are 0..3, b's 4..7)
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
// Queries against an FP8 key page: the head dims are taken in a permuted order
// shared by queries and keys (a dot product does not depend on the order), so
// that in MMA step kk lane q supplies physical dims 16*(2q + kk/4) + 4*(kk%4) + j
// from one 4-byte word of a key row.  Logical column (in the f16 query rows the
// A fragments are loaded from) of physical head dim p:
__device__ __forceinline__ int q_col_fp8(int p) {
    const int kk = 4 * ((p >> 4) & 1) + ((p >> 2) & 3), q = p >> 5, j = p & 3;
    return 16 * kk + 2 * q + (j & 1) + 8 * (j >> 1);
}
// eight FP4 E2M1 codes (byte i of v holds codes 2i, 2i+1, low nibble first)
// -> four f16x2 words, d_i from byte i
__device__ __forceinline__ void e2m1x8_f16(uint32_t v, uint32_t &d0, uint32_t &d1, uint32_t &d2, uint32_t &d3) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
        : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
        : "r"(v));
}
__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// 2^d in both halves of an f16x2 word, d <= 0 (subnormal below 2^-14, 0 below 2^-24)
__device__ __forceinline__ uint32_t pow2_f16x2(int d) {
    const uint32_t h = d >= -14 ? (uint32_t)(15 + d) << 10 : d >= -24 ? 1u << (24 + d) : 0u;
    return h | (h << 16);
}
// value of an E8M0 scale byte: 2^(e - 127) (0: 2^-127, 255: NaN)
__device__ __forceinline__ float e8m0_f(int e) {
    return e == 0 ? __uint_as_float(0x00400000u) : e == 255 ? __uint_as_float(0x7fc00000u) : __uint_as_float((uint32_t)e << 23);
}
// two bf16 (low half first) -> f16x2
__device__ __forceinline__ uint32_t bf16x2_f16x2(uint32_t v) {
    float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xffff0000u);
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
// Fixed-point (2^-32) conversions.  The 64-bit integer <-> float conversion
// instructions issue on the FP64 pipe, which on this part runs at a small
// fraction of the integer and FP32 rate, so both directions are built from
// 32-bit operations.
// to_fx: |v| * 2^32 rounded half away from zero, from the float's fields
// (|v| < 2^31; zero and subnormal inputs give 0).
__device__ __forceinline__ long long to_fx(float v) {
    const uint32_t b = __float_as_uint(v);
    const int e = (int)((b >> 23) & 0xffu);
    const uint32_t m = (b & 0x7fffffu) | 0x800000u;
    const int s = e - 118;  // |v| * 2^32 = m * 2^(e - 118)
    unsigned long long r;
    if (s >= 0) r = (unsigned long long)m << min(s, 39);
    else if (s > -25) r = (m + (1u << (-s - 1))) >> (-s);
    else r = 0;
    if (e == 0) r = 0;
    return (b >> 31) ? -(long long)r : (long long)r;
}
// exact float of an integer u < 2^23: u is placed in the significand of 2^23
// and 2^23 subtracted (FP32 and logic pipes only)
__device__ __forceinline__ float u23_to_f(uint32_t u) {
    return __uint_as_float(0x4b000000u | u) - 8388608.0f;
}
// from_fx: the magnitude's bits in three pieces of at most 22 bits, each
// converted exactly, recombined with two fused multiply-adds (|v| < 2^63)
__device__ __forceinline__ float from_fx(long long v) {
    const unsigned long long a = v < 0 ? 0ull - (unsigned long long)v : (unsigned long long)v;
    const uint32_t lo = (uint32_t)a, hi = (uint32_t)(a >> 32);
    const float f0 = u23_to_f(lo & 0x3fffffu);
    const float f1 = u23_to_f((lo >> 22) | ((hi & 0xfffu) << 10));
    const float f2 = u23_to_f(hi >> 12);
    const float f = fmaf(f2, 4096.0f, fmaf(f1, 1.0f / 1024.0f, f0 * (1.0f / MK_FX)));
    return v < 0 ? -f : f;
}
__device__ __forceinline__ void red_add(long long *p, long long v) {
    atomicAdd(reinterpret_cast<unsigned long long *>(p), (unsigned long long)v);
}
// arrival at a counter with release semantics at GPU scope: every write this
// CTA made before the preceding CTA barrier is visible to a thread whose
// acquire load sees the new count (the barrier orders the other threads'
// writes before this thread's release)
__device__ __forceinline__ void arrive_release(unsigned long long *p) {
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(p) : "memory");
}
__device__ __forceinline__ void arrive_release(int *p) {
    asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p) : "memory");
}
__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// byte address of (row, byte) inside a TMA box stored with the 128-byte swizzle
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int byte) {
    return base + row * 128 + ((((byte >> 4) ^ (row & 7)) << 4) | (byte & 15));
}

// ------------------------------------------------------------------ CTA context
// input blocks of this CTA's fragment builds, fixed for the launch: the QKV
// stage's (and those it stores sum-of-squares partials for), the O
// projection's, the router stage's (and its partials)
enum { KBM_QKV = 0, KBM_QKV_SSQ, KBM_O, KBM_RT, KBM_RT_SSQ };
// The integer state with which a CTA starts walking its tiles of one GEMV
// stage (see StageIter): its tile count and the (expert slot, matrix, row
// group, column piece) of its first tile.  Working it out takes a chain of
// integer divisions; the stages whose split is fixed for the launch get it once
// at launch, the routed stages once per layer while the routing is published.
struct StageSeed {
    int n, ex, mat, rg, kc, kc0, kcn, kcn_sh, n_rg, n_kc, nmat, nex, nd;
};
struct RouteSm {
    int nd;
    int dlist[MK_MAXD];
    signed char dslot[MK_MAXD][MK_MAXT];
    int idx[MK_MAXT][MK_MAXK];
    float w[MK_MAXT][MK_MAXK];
    StageSeed seed[2];           // this CTA's routed gate/up and down stages
};
// CTA-uniform state in shared memory: the model block and the current/next
// layer's descriptors are copied here so that no stage reads them from global
// memory, and the per-thread context can be rebuilt in registers anywhere.
struct MiscSm {
    int abort;
    int gs_ok;
    int emask[16];               // routed experts of the block (bit set)
    int epre[16];                // routed experts in the mask words before each word
    float inv_rms[3][MK_MAXT];   // attention, moe, final
    int distinct_total;
    int valid, ctx, nsplit;
    int nbar;                    // grid barriers passed (thread 0)
    int nmark;                   // trace events written (thread 0)
    int par;                     // parity of the current layer: selects its accumulators
    unsigned long long base;     // barrier counter at launch
    const Params *p;             // points at pc below
    DModel m;
    DLayer L[2];                 // descriptors of layers with parity 0 / 1
    StageSeed seed[8];           // this CTA's split of the stages fixed for the launch, by stage
    uint32_t kbm[5];             // 128-column input blocks of the fragment builds (see KBM_*)
    Params pc;                   // the launch parameters: generic loads from the
                                 // kernel's parameter space are slow, shared memory is not
};

struct Ctx {
    const Params *p;
    const DModel *m;             // shared-memory copy
    Ctrl *ctrl;
    unsigned char *sm;
    uint64_t *full, *empty, *route;
    RouteSm *rt;          // [2]
    MiscSm *misc;
    int cta, G, T, ctx, nsplit, tid, warp, lane;
    long long timeout;
    bool prof;
};

static_assert(sizeof(MiscSm) <= SM_MISC_BYTES, "shared-memory context block too large");
static_assert(sizeof(RouteSm) * 2 <= SM_ROUTE_BYTES, "routing block too large");

__device__ __forceinline__ unsigned char *smem_base() {
    extern __shared__ unsigned char smem_raw[];
    // the 128-byte TMA swizzle pattern repeats every 1024 bytes: align the map to it
    return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
}
// the context of the calling thread, from special registers and shared memory
__device__ __forceinline__ Ctx make_ctx() {
    Ctx c;
    c.sm = smem_base();
    c.misc = reinterpret_cast<MiscSm *>(c.sm + SM_MISC);
    c.p = c.misc->p;
    c.m = &c.misc->m;
    c.ctrl = c.m->ctrl;
    c.full = reinterpret_cast<uint64_t *>(c.sm + SM_BAR);
    c.empty = c.full + MK_RING;
    c.route = c.empty + MK_RING;
    c.rt = reinterpret_cast<RouteSm *>(c.sm + SM_ROUTE);
    c.cta = blockIdx.x;
    c.G = gridDim.x;
    c.T = c.p->T;
    c.ctx = c.misc->ctx;
    c.nsplit = c.misc->nsplit;
    c.tid = threadIdx.x;
    c.warp = threadIdx.x >> 5;
    c.lane = threadIdx.x & 31;
    c.timeout = c.m->timeout_ns;
    c.prof = c.p->marks != nullptr;
    return c;
}

// intra-stage trace event (thread 0 of the consumers, only when tracing).
// Helpers that run at many call sites but rarely or off the hot loop are kept
// out of line: most of the step's code runs once per layer, so every inlined
// copy is code the instruction cache fetches again each layer.
__device__ __noinline__ void mark_slow(int id) {
    const Ctx c = make_ctx();
    const Params &p = *c.p;
    const int k = c.misc->nmark;
    if (k < MK_MARKS - 80) {
        unsigned long long *e = p.marks + ((long long)c.cta * MK_MARKS + k) * 2;
        e[0] = (unsigned long long)id;
        e[1] = gtimer();
    }
    c.misc->nmark = k + 1;
}
__device__ __forceinline__ void mark(const Ctx &c, int id) {
    if (c.prof && c.tid == 0) mark_slow(id);
}

// trace value written at a fixed event slot (cycle counts of a loop)
__device__ __forceinline__ void mark_val(const Ctx &c, int slot, int id, unsigned long long v) {
    const Params &p = *c.p;
    if (p.marks && slot < MK_MARKS) {
        unsigned long long *e = p.marks + ((long long)c.cta * MK_MARKS + slot) * 2;
        e[0] = (unsigned long long)id;
        e[1] += v;
    }
}

// abort flag of this CTA (shared memory).  Only the grid-barrier thread reads
// the device-wide flag and mirrors it here, so waiting threads never poll
// global memory for it.
__device__ __forceinline__ bool aborted(const Ctx &c) {
    return *(volatile int *)&c.misc->abort != 0;
}
__device__ __forceinline__ bool aborted_global(const Ctx &c) {
    if (*(volatile int *)&c.ctrl->abort != 0) *(volatile int *)&c.misc->abort = 1;
    return aborted(c);
}
__device__ void raise_err(const Ctx &c, int code, int where) {
    *(volatile int *)&c.misc->abort = 1;
    if (atomicCAS(&c.ctrl->status, 0, code) == 0) atomicExch(&c.ctrl->where, where);
    atomicExch(&c.ctrl->abort, 1);
}
// a value left the range of the kernel's number formats: an f16 GEMV input
// beyond 65504 (or NaN), a rotated query beyond it (f16 queries of the FP8 KV
// attention), or a partial sum of magnitude 2^31 or more that the
// 2^-32 fixed-point accumulators cannot hold.  The step stops with MK_ERR_RANGE
// instead of returning infinities or wrapped sums.
__device__ __noinline__ void range_err(int where) {
    const Ctx c = make_ctx();
    raise_err(c, MK_ERR_RANGE, where);
}
// nonzero if either half of an f16x2 word is infinite or NaN (exponent all ones)
__device__ __forceinline__ uint32_t f16x2_bad(uint32_t w) {
    return __vcmpeq2(w & 0x7c007c00u, 0x7c007c00u);
}
// nonzero unless |v| < 2^31 (NaN included)
__device__ __forceinline__ uint32_t fx_bad(float v) { return !(fabsf(v) < 2147483648.0f); }

// bounded wait on an mbarrier phase, spun inline (no call on the path whose
// length depends on timing)
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity, const Ctx &c, int where) {
    if (mbar_try(b, parity)) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(b, parity)) return true;
        if ((it & 15) == 0) {
            if (aborted(c)) return false;
            if ((long long)(gtimer() - t0) > c.timeout) {
                raise_err(c, MK_ERR_TIMEOUT, where);
                return false;
            }
        }
    }
}
// bounded wait that ignores the abort flag (drain of copies in flight)
__device__ void mbar_wait_drain(uint64_t *b, uint32_t parity, const Ctx &c) {
    uint64_t t0 = gtimer();
    while (!mbar_try(b, parity)) {
        if ((long long)(gtimer() - t0) > c.timeout) return;
    }
}
// spins of one thread on a counter in global memory.  Each poll is one
// acquire load that waits for its answer, so a CTA keeps at most one request
// to the line in flight; a sleep between polls (64 ns) measured no better.
// Timeout and abort are checked every 16 polls.
__device__ bool spin_ge_u64(unsigned long long *a, unsigned long long target, const Ctx &c,
                            int where) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
        if (v >= target) return true;
        if ((it & 15) == 15) {
            if (aborted_global(c)) return false;
            uint64_t now = gtimer();
            if (t0 == 0) t0 = now;
            else if ((long long)(now - t0) > c.timeout) {
                raise_err(c, MK_ERR_TIMEOUT, where);
                return false;
            }
        }
    }
}
__device__ bool spin_ge_s32(int *a, int target, const Ctx &c, int where) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        int v;
        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
        if (v >= target) return true;
        if ((it & 15) == 15) {
            if (aborted_global(c)) return false;
            uint64_t now = gtimer();
            if (t0 == 0) t0 = now;
            else if ((long long)(now - t0) > c.timeout) {
                raise_err(c, MK_ERR_TIMEOUT, where);
                return false;
            }
        }
    }
}

// grid-wide barrier among the consumer warps of all CTAs; split into arrive/wait
__device__ __noinline__ void grid_arrive_nc() {
    const Ctx c = make_ctx();
    bar_consumers();
    if (c.tid == 0) {
        const int nbar = ++c.misc->nbar;
        const Params &p = *c.p;
        if (p.stage_trace && nbar <= p.stage_cap)
            p.stage_trace[((long long)c.cta * p.stage_cap + nbar - 1) * 2] = gtimer();
        // test hook (mk_debug_skip_barrier): CTA 0 withholds one arrival so that
        // every other CTA's bounded wait runs out
        if (!(p.skip_barrier == nbar && c.cta == 0)) arrive_release(&c.ctrl->bar_count);
    }
}
__device__ __noinline__ bool grid_wait_nc(int where) {
    const Ctx c = make_ctx();
    if (c.tid == 0) {
        const int nbar = c.misc->nbar;
        // the abort flag is read alongside the first poll, not before it; the
        // acquire loads of the poll order every later read of other CTAs' data
        // (all of which goes through L2) after their arrivals
        const int ab = *(volatile int *)&c.ctrl->abort;
        bool ok = spin_ge_u64(&c.ctrl->bar_count, c.misc->base + (unsigned long long)nbar * c.G, c, where);
        if (ab) *(volatile int *)&c.misc->abort = 1;
        c.misc->gs_ok = ok && !aborted(c);
        const Params &p = *c.p;
        if (p.stage_trace && nbar <= p.stage_cap)
            p.stage_trace[((long long)c.cta * p.stage_cap + nbar - 1) * 2 + 1] = gtimer();
    }
    bar_consumers();
    return c.misc->gs_ok != 0;
}
__device__ __forceinline__ void grid_arrive(const Ctx &c) {
    (void)c;
    grid_arrive_nc();
}
__device__ __forceinline__ bool grid_wait(const Ctx &c, int where) {
    (void)c;
    return grid_wait_nc(where);
}
__device__ __forceinline__ bool grid_sync(const Ctx &c, int where) {
    grid_arrive(c);
    return grid_wait(c, where);
}

// ------------------------------------------------------------------ schedules
// the products stay below 2^32 for every split this kernel makes (at most
// 8 x 129,280 elements over 152 parts), so 32-bit unsigned arithmetic is exact
__device__ __forceinline__ void split_range(int total, int parts, int part, int &b, int &e) {
    b = (int)((unsigned)total * (unsigned)part / (unsigned)parts);
    e = (int)((unsigned)total * (unsigned)(part + 1) / (unsigned)parts);
}

// Per-layer accumulators come in two copies selected by the layer's parity, so
// that the copy the next layer uses can be cleared while this layer runs.
enum { ACC_QKV = 0, ACC_SH, ACC_EA, ACC_RLOG };
__device__ __forceinline__ long long acc_elems(const DModel &m, int which) {
    return which == ACC_QKV ? (long long)MK_MAXT * m.nqkv
         : which == ACC_SH ? (long long)MK_MAXT * 2 * m.I
         : which == ACC_EA ? (long long)MK_MAXT * m.K * 2 * m.I : (long long)MK_MAXT * m.E;
}
__device__ __forceinline__ long long *acc_ptr(const DModel &m, int which, int par) {
    long long *b = which == ACC_QKV ? m.qkv_acc : which == ACC_SH ? m.sh_acc : which == ACC_EA ? m.ea_acc : m.rlog;
    return b + (par ? acc_elems(m, which) : 0);
}



// attention split of a unit (one kv head, a run of pages)
struct AttUnit {
    bool active, has_new;
    int g, s, p0, pc1;
};
__device__ AttUnit att_unit(const Ctx &c) {
    const DModel &m = *c.m;
    AttUnit u;
    int ncp = (c.ctx + m.P - 1) / m.P, np = ncp + 1;
    u.active = c.cta < m.Hkv * c.nsplit;
    u.g = c.cta / c.nsplit;
    u.s = c.cta - u.g * c.nsplit;
    int p1;
    split_range(np, c.nsplit, u.s, u.p0, p1);
    u.pc1 = min(p1, ncp);
    u.has_new = (p1 == np);
    return u;
}

// register copy of the matrix-descriptor fields the tile loops use
struct MatR {
    const CUtensorMap *tmap;
    const float *scale;
    const CUtensorMap *smap;
    long long sest;
    int rows, cols, xstep, dtype, is3d;
};
__device__ __forceinline__ MatR mat_regs(const DMat &d) {
    MatR r;
    r.tmap = d.tmap;
    r.scale = d.scale;
    r.smap = d.smap;
    r.sest = d.scale_estride;
    r.rows = d.rows;
    r.cols = d.cols;
    r.xstep = d.es ? 128 / d.es : 128;
    r.dtype = d.dtype;
    r.is3d = d.is3d;
    return r;
}

// Walks the tiles of one stage that belong to this CTA, in (expert slot,
// matrix, 128-row group, 128-byte column chunk) order.  Descriptors are read
// once per stage; the position advances with counters, no divisions.
// Walks the tiles of one stage that belong to this CTA.  The router, shared
// gate/up and routed gate/up stages are ordered column chunk first (1024
// input columns), then (expert slot, matrix, 256-row group, 128-byte column
// piece): every CTA then works inside one or two chunks and needs only those
// columns of its input.  Other stages are one chunk wide.  Descriptors are
// read once per stage; the position advances with counters, no divisions.
struct StageIter {
    MatR m0, m1;          // matrix 0 / 1 (gate/up pairs; routed/shared down)
    int n_rg, n_kc, nmat, nex, nd;
    int ex, mat, rg, kc, n;
    int kc0, kcn;         // first column piece of the current chunk; pieces per chunk
    int kcn_sh;           // down projections: pieces per row group of the shared expert
    int st;
    const int *dlist;
    __device__ __forceinline__ const MatR &cur() const {
        return (st == ST_EXPB ? ex >= nd : mat != 0) ? m1 : m0;
    }
    __device__ __forceinline__ int expert() const {
        return (st == ST_EXPA || (st == ST_EXPB && ex < nd)) ? dlist[ex] : 0;
    }
    __device__ __forceinline__ bool item_start() const { return kc == kc0; }
    __device__ __forceinline__ void advance() {
        if (++kc == kc0 + kcn) {
            kc = kc0;
            if (++rg == n_rg) {
                rg = 0;
                if (++mat == nmat) {
                    mat = 0;
                    if (++ex == nex) {
                        ex = 0;
                        kc0 += kcn;
                        kc = kc0;
                    } else if (ex == nd && st == ST_EXPB) {
                        kcn = kcn_sh;  // the shared expert may be stored in another format
                    }
                }
            }
        }
    }
};

__device__ __forceinline__ bool chunk_major(int st) { return st == ST_ROUTER || st == ST_SHA || st == ST_EXPA; }

// 128-column blocks of the input chunks this CTA works on in the chunk-major
// stages (input width `cols`): chunks nch*cta/G .. ceil(nch*(cta+1)/G) - 1,
// whatever the number of tiles per chunk
__device__ uint32_t chunk_kb_mask(const Ctx &c, int cols) {
    const uint32_t all = 0xffffffffu >> (32 - cols / 128);
    if (cols % 1024) return all;
    const int nch = cols / 1024;
    const int c0 = nch * c.cta / c.G, c1 = (nch * (c.cta + 1) + c.G - 1) / c.G - 1;
    uint32_t msk = 0;
    for (int ch = c0; ch <= c1 && ch < nch; ++ch) msk |= 0xffu << (8 * ch);
    return msk & all;
}

// blocks whose sum-of-squares partial this CTA stores in the chunk-major
// stages: the first CTA of each chunk takes that chunk's blocks (CTA 0 takes
// every block when the input is not cut into chunks)
__device__ uint32_t ssq_owner_mask(const Ctx &c, int cols) {
    const uint32_t all = 0xffffffffu >> (32 - cols / 128);
    if (cols % 1024) return c.cta == 0 ? all : 0u;
    const int nch = cols / 1024, c0 = nch * c.cta / c.G;
    if (c.cta > 0 && nch * (c.cta - 1) / c.G == c0) return 0u;
    return (0xffu << (8 * c0)) & all;
}

// this CTA's split of stage st (nd: routed experts of the layer, for the
// routed stages).  Every layer of a model has the same matrix shapes, so the
// split of the non-routed stages holds for the whole launch.
__device__ void stage_seed(StageSeed &sd, const Ctx &c, int st, const DLayer &L, int nd) {
    const DModel &m = *c.m;
    sd.nmat = 1;
    sd.nex = 1;
    sd.nd = 0;
    if (st == ST_SHA) {
        sd.nmat = 2;
        sd.nex = m.nshared;
    } else if (st == ST_EXPA) {
        sd.nmat = 2;
        sd.nex = nd;
        sd.nd = nd;
    } else if (st == ST_EXPB) {
        sd.nd = nd;
        sd.nex = nd + m.nshared;
    }
    const DMat &d0 = st == ST_QKV ? L.qkv : st == ST_O ? L.o : st == ST_ROUTER ? L.router :
                     st == ST_LM ? m.lm : st == ST_SHA ? L.s1 : st == ST_EXPA ? L.w1 : L.w2;
    sd.n_rg = d0.n_rg;
    sd.n_kc = d0.n_kc;
    sd.kcn = (chunk_major(st) && d0.cols % 1024 == 0) ? 1024 / d0.cpk : sd.n_kc;
    if (st == ST_EXPB) {
        // items (expert slot, 256-row group), whole items per CTA as below; the
        // shared expert's items have its own number of column pieces (MXFP4
        // routed experts: 256 columns a piece, an FP8 shared expert: 128)
        const int kr = sd.kcn, ks = m.nshared ? L.s2.n_kc : kr, nrt = sd.nd * sd.n_rg;
        sd.kcn_sh = ks;
        int bi, ei;
        split_range(sd.nex * sd.n_rg, c.G, c.cta, bi, ei);
        sd.n = (min(ei, nrt) - min(bi, nrt)) * kr + (max(ei, nrt) - max(bi, nrt)) * ks;
        sd.ex = bi / sd.n_rg;
        sd.rg = bi - sd.ex * sd.n_rg;
        sd.mat = 0;
        sd.kc0 = sd.kc = 0;
        if (sd.ex >= sd.nd) sd.kcn = ks;
        return;
    }
    sd.kcn_sh = sd.kcn;
    const int nch = sd.n_kc / sd.kcn;
    const int per_mat = sd.n_rg * sd.kcn, per_ex = sd.nmat * per_mat, per_ch = sd.nex * per_ex;
    int b, e;
    if (st == ST_EXPA) {
        // whole items only: an item's partial sum is then formed by one CTA in
        // a fixed tile order whatever the number of routed experts, so the
        // step's result for a token does not depend on the other tokens of
        // the block (batch invariance); per-CTA counts differ by one item
        split_range(nch * per_ch / sd.kcn, c.G, c.cta, b, e);
        b *= sd.kcn;
        e *= sd.kcn;
    } else {
        split_range(nch * per_ch, c.G, c.cta, b, e);
    }
    sd.n = e - b;
    const int ch = per_ch ? b / per_ch : 0;
    int r = b - ch * per_ch;
    sd.ex = per_ex ? r / per_ex : 0;
    r -= sd.ex * per_ex;
    sd.mat = per_mat ? r / per_mat : 0;
    r -= sd.mat * per_mat;
    sd.rg = r / sd.kcn;
    sd.kc0 = ch * sd.kcn;
    sd.kc = sd.kc0 + (r - sd.rg * sd.kcn);
}

// start walking this CTA's tiles of stage st: the layer's matrix descriptors
// and the split worked out beforehand (the launch's for the non-routed stages,
// the layer's routing for the routed ones)
__device__ __forceinline__ void stage_iter(StageIter &it, const Ctx &c, int st, const DLayer &L, const RouteSm *rt) {
    const DModel &m = *c.m;
    it.st = st;
    it.dlist = rt->dlist;
    switch (st) {
        case ST_QKV: it.m0 = mat_regs(L.qkv); break;
        case ST_O: it.m0 = mat_regs(L.o); break;
        case ST_ROUTER: it.m0 = mat_regs(L.router); break;
        case ST_LM: it.m0 = mat_regs(m.lm); break;
        case ST_SHA:
            it.m0 = mat_regs(L.s1);
            it.m1 = mat_regs(L.s3);
            break;
        case ST_EXPA:
            it.m0 = mat_regs(L.w1);
            it.m1 = mat_regs(L.w3);
            break;
        default:  // ST_EXPB
            it.m0 = mat_regs(L.w2);
            it.m1 = mat_regs(L.s2);
            break;
    }
    const StageSeed &sd = st == ST_EXPA ? rt->seed[0] : st == ST_EXPB ? rt->seed[1] : c.misc->seed[st];
    it.n = sd.n;
    it.ex = sd.ex;
    it.mat = sd.mat;
    it.rg = sd.rg;
    it.kc = sd.kc;
    it.kc0 = sd.kc0;
    it.kcn = sd.kcn;
    it.kcn_sh = sd.kcn_sh;
    it.n_rg = sd.n_rg;
    it.n_kc = sd.n_kc;
    it.nmat = sd.nmat;
    it.nex = sd.nex;
    it.nd = sd.nd;
}

// ------------------------------------------------------------------ producer
// MK_PLANES lanes of the producer warp issue copies side by side: lane j takes
// the stage's tiles j, j + MK_PLANES, ...  With MK_PLANES == MK_RING every lane
// owns one ring slot, so four tiles are requested concurrently while each lane
// keeps its own wait -> arm -> copy chain.

// producer-side state of one issuing lane (registers of the producer)
struct Prod {
    uint64_t pol;                 // L2 evict-first policy of streamed weights and KV pages
    uint32_t pi;                  // ring positions handed out so far
    int last;                     // last position this lane armed (-1: none)
    unsigned long long wait, tma, bulk;
};

// wait for ring position pos to be free and arm its full barrier for `bytes`
__device__ __forceinline__ bool prod_take(const Ctx &c, Prod &ps, uint32_t pos, uint32_t bytes) {
    const uint32_t slot = pos % MK_RING;
    unsigned long long cy1 = c.prof ? clock64() : 0;
    if (!mbar_wait(&c.empty[slot], ((pos / MK_RING) & 1) ^ 1, c, 100)) return false;
    if (c.prof) ps.wait += clock64() - cy1;
    mbar_expect_tx(&c.full[slot], bytes);
    ps.last = (int)pos;
    return true;
}



__device__ __forceinline__ bool prod_gemv_impl(const Ctx &c, Prod &ps, int st, const DLayer &L,
                                               const RouteSm *rt) {
    StageIter it;
    stage_iter(it, c, st, L, rt);
    const int n = it.n;
    for (int j = 0; j < c.lane && j < n; ++j) it.advance();
    unsigned char *const ring = c.sm + SM_RING, *const sbase = c.sm + SM_SCALE;
    uint64_t *const full = c.full;
    bool ok = true;
    for (int t = c.lane; t < n; t += MK_PLANES) {
        const MatR &d = it.cur();
        const int e = it.expert();
        uint32_t sbytes = 0;
        if (d.dtype == MK_DT_FP8E4M3_B128) sbytes = min(256, d.rows - it.rg * 256) * 4;
        else if (d.dtype == MK_DT_MXFP4_B32) sbytes = 8 * 256;  // one box of E8M0 scales
        const uint32_t pos = ps.pi + t, slot = pos % MK_RING;
        if (!prod_take(c, ps, pos, MK_SLOT + sbytes)) {
            ok = false;
            break;
        }
        void *dst = ring + slot * MK_SLOT;
        const int x = it.kc * d.xstep, y = it.rg * 256;
        unsigned long long t0 = c.prof ? clock64() : 0;
        if (d.is3d) tma3d_h(dst, d.tmap, x, y, e, &full[slot], ps.pol);
        else tma2d_h(dst, d.tmap, x, y, &full[slot], ps.pol);
        unsigned long long t1 = c.prof ? clock64() : 0;
        if (d.dtype == MK_DT_MXFP4_B32) {
            // scales [E][cols/32][rows]: the tile's 8 groups x 256 rows
            if (d.is3d) tma3d_h(sbase + slot * MK_SCALE_SLOT, d.smap, y, it.kc * 8, e, &full[slot], ps.pol);
            else tma2d_h(sbase + slot * MK_SCALE_SLOT, d.smap, y, it.kc * 8, &full[slot], ps.pol);
        } else if (sbytes) {
            const float *src = d.scale + (long long)e * d.sest + (long long)it.kc * d.rows + y;
            bulk_g2s_h(sbase + slot * MK_SCALE_SLOT, src, sbytes, &full[slot], ps.pol);
        }
        if (c.prof) {
            unsigned long long t2 = clock64();
            ps.tma += t1 - t0;
            ps.bulk += t2 - t1;
        }
#pragma unroll
        for (int j = 0; j < MK_PLANES; ++j) it.advance();
    }
    ps.pi += n;
    // every lane has issued its tiles of this stage before any lane starts the
    // next one, so no slot's empty barrier is ever waited on two phases ahead
    return __all_sync((1u << MK_PLANES) - 1, ok);
}

__device__ __noinline__ bool prod_gemv(const Ctx &c, Prod &ps, int st, const DLayer &L, const RouteSm *rt) {
    const bool prof = c.prof && c.lane == 0;
    unsigned long long cy0 = prof ? clock64() : 0, w0 = ps.wait, a0 = ps.tma, b0 = ps.bulk;
    bool ok = prod_gemv_impl(c, ps, st, L, rt);
    if (prof) {
        mark_val(c, MK_MARKS - 32 + st * 2 + 0, 950 + st * 2 + 0, ps.wait - w0);
        mark_val(c, MK_MARKS - 32 + st * 2 + 1, 950 + st * 2 + 1, clock64() - cy0);
        mark_val(c, MK_MARKS - 16 + st * 2 + 0, 980 + st * 2 + 0, ps.tma - a0);
        mark_val(c, MK_MARKS - 16 + st * 2 + 1, 980 + st * 2 + 1, ps.bulk - b0);
    }
    return ok;
}

// this CTA's KV pages of one layer: K in the first half of a slot, V in the second
__device__ __forceinline__ bool prod_att(const Ctx &c, Prod &ps, int l) {
    const DModel &m = *c.m;
    AttUnit u = att_unit(c);
    if (!u.active) return true;  // uniform across the producer lanes
    const int nbox = (m.d * m.kv_es) / 128;
    const CUtensorMap *km = c.p->kvmaps + 2 * l, *vm = km + 1;
    bool ok = true;
    for (int j = u.p0 + c.lane; j < u.pc1; j += MK_PLANES) {
        const int phys = __ldg(c.p->page_table + j);
        const int y = (phys * m.Hkv + u.g) * m.P;
        const uint32_t pos = ps.pi + (j - u.p0);
        if (!prod_take(c, ps, pos, 2 * nbox * m.P * 128)) {
            ok = false;
            break;
        }
        unsigned char *dst = c.sm + SM_RING + (pos % MK_RING) * MK_SLOT;
        uint64_t *bar = &c.full[pos % MK_RING];
        for (int bx = 0; bx < nbox; ++bx) {
            tma2d_h(dst + bx * m.P * 128, km, bx * (128 / m.kv_es), y, bar, ps.pol);
            tma2d_h(dst + MK_SLOT / 2 + bx * m.P * 128, vm, bx * (128 / m.kv_es), y, bar, ps.pol);
        }
    }
    ps.pi += u.pc1 - u.p0;
    return __all_sync((1u << MK_PLANES) - 1, ok);
}

// lanes 0..MK_PLANES-1 of the producer warp
__device__ __noinline__ void producer() {
    const Ctx c = make_ctx();
    const DModel &m = *c.m;
    const Params &p = *c.p;
    Prod ps;
    ps.pol = l2_evict_first();
    ps.pi = 0;
    ps.last = -1;
    ps.wait = ps.tma = ps.bulk = 0;
    int nl = p.mode ? 1 : m.L;
    bool ok = true;
    for (int li = 0; li < nl && ok; ++li) {
        int l = p.mode ? p.layer : li;
        const DLayer &L = c.misc->L[li & 1];
        const RouteSm *rt = &c.rt[li & 1];
        ok = prod_gemv(c, ps, ST_QKV, L, rt) && prod_att(c, ps, l) && prod_gemv(c, ps, ST_O, L, rt) &&
             prod_gemv(c, ps, ST_ROUTER, L, rt) && prod_gemv(c, ps, ST_SHA, L, rt);
        if (!ok) break;
        ok = __all_sync((1u << MK_PLANES) - 1, mbar_wait(c.route, li & 1, c, 101));
        if (!ok) break;
        ok = prod_gemv(c, ps, ST_EXPA, L, rt) && prod_gemv(c, ps, ST_EXPB, L, rt);
    }
    if (ok && p.mode == 0) ok = prod_gemv(c, ps, ST_LM, c.misc->L[0], &c.rt[0]);
    // after a failure every copy this lane may still have in flight must land
    // before the CTA exits: those are the last MK_RING armed ring positions (a
    // slot is re-armed only after its previous copy completed and was consumed;
    // a position whose copy already landed passes its wait at once)
    if (!ok && ps.last >= 0)
        for (int pos = max(0, ps.last - (MK_RING - 1)); pos <= ps.last; ++pos)
            mbar_wait_drain(&c.full[pos % MK_RING], (pos / MK_RING) & 1, c);
}

// ------------------------------------------------------------------ activations
// Fragment order of the B operand (activations) of one 128-column block: for
// step s (0..7) and lane l = 4n + q the lane holds token n's columns
//   32q + 8*(((s>>1) + 2*(q>>1)) & 3) + 4*(s&1) + j,  j = 0..3,
// as two f16x2 words.  The weight side reads the same columns (a permutation of
// the reduction index shared by both operands), which lets every lane fetch its
// FP8/bf16 weights as whole 16-byte swizzled chunks without bank conflicts.
__device__ __forceinline__ int frag_col(int s, int q, int j) {
    return 32 * q + 8 * (((s >> 1) + 2 * (q >> 1)) & 3) + 4 * (s & 1) + j;
}

// source of a GEMV input: fixed-point [T][stride] times gamma, or float [T][stride]
struct ActSrc {
    const long long *fx;
    const float *f32;
    int stride;
    const float *gamma;
};
// four consecutive activation values from column col (col % 4 == 0)
__device__ __forceinline__ float4 act4(const ActSrc &a, int t, int col) {
    float4 v;
    if (a.fx) {
        const longlong2 *p = reinterpret_cast<const longlong2 *>(a.fx + (long long)t * a.stride + col);
        longlong2 x = __ldcg(p), y = __ldcg(p + 1);
        v = make_float4(from_fx(x.x), from_fx(x.y), from_fx(y.x), from_fx(y.y));
    } else {
        v = __ldcg(reinterpret_cast<const float4 *>(a.f32 + (long long)t * a.stride + col));
    }
    if (a.gamma) {
        float4 g = __ldg(reinterpret_cast<const float4 *>(a.gamma + col));
        v.x *= g.x;
        v.y *= g.y;
        v.z *= g.z;
        v.w *= g.w;
    }
    return v;
}

// byte offset, in the fragment buffer, of columns 4*c4 .. 4*c4+3 (c4 < 32) of
// 128-column block kb for token t (the inverse of frag_col)
__device__ __forceinline__ uint32_t frag_off(int kb, int t, int c4) {
    const int q = c4 >> 3, sb = c4 & 1, x = (c4 >> 1) & 3;
    return kb * 2048 + ((((x - 2 * (q >> 1)) & 3) * 32 + 4 * t + q) << 4) + sb * 8;
}
// build f16 fragments for the 128-column blocks in `mask` (consumer threads).
// Thread (t, c4) = (tid / 32, tid % 32) converts columns 4*c4 .. 4*c4+3 of
// token t in every block, so each warp reads one token's block row as whole
// contiguous L2 lines.
// Tokens t >= T get zeros (the MMA reduces against all eight token columns).
// Four blocks are in flight before any is converted.
// Blocks in ssq_mask (a subset of mask, residual input only) also get their
// RMSNorm sum-of-squares partial: warp t sums token t's 128 values of the
// block (before gamma) and stores it as ssq[which][kb][t].
__device__ __noinline__ void build_frags(const ActSrc a, uint32_t mask, uint32_t ssq_mask = 0, int which = 0) {
    const Ctx c = make_ctx();
    unsigned char *fr = c.sm + SM_SCRATCH;
    const int t = c.tid >> 5, c4 = c.lane;
    const bool live = t < c.T;
    const long long *fx = a.fx ? a.fx + (long long)t * a.stride + 4 * c4 : nullptr;
    const float *f32 = a.f32 ? a.f32 + (long long)t * a.stride + 4 * c4 : nullptr;
    const float *gm = a.gamma ? a.gamma + 4 * c4 : nullptr;
    const uint32_t o_tc = frag_off(0, t, c4);
    constexpr int B = 4;  // blocks in flight per thread (8 measured slower: register pressure)
    uint32_t rest = mask, bad = 0;
    while (rest) {
        int kb[B];
        longlong2 x0[B], x1[B];
        float4 xf[B], g[B];
#pragma unroll
        for (int u = 0; u < B; ++u) {
            kb[u] = rest ? __ffs(rest) - 1 : -1;
            rest &= rest - 1;
            x0[u] = x1[u] = make_longlong2(0, 0);
            xf[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            g[u] = make_float4(1.f, 1.f, 1.f, 1.f);
            if (kb[u] >= 0 && live) {
                const int col = kb[u] * 128;
                if (fx) {  // one 256-bit load (the 32 bytes are 32-byte aligned)
                    long long v0, v1, v2, v3;
                    asm volatile("ld.global.cg.v4.b64 {%0,%1,%2,%3}, [%4];"
                                 : "=l"(v0), "=l"(v1), "=l"(v2), "=l"(v3)
                                 : "l"(fx + col));
                    x0[u] = make_longlong2(v0, v1);
                    x1[u] = make_longlong2(v2, v3);
                } else {
                    xf[u] = __ldcg(reinterpret_cast<const float4 *>(f32 + col));
                }
                if (gm) g[u] = __ldg(reinterpret_cast<const float4 *>(gm + col));
            }
        }
#pragma unroll
        for (int u = 0; u < B; ++u) {
            if (kb[u] < 0) break;
            const float4 v = fx ? make_float4(from_fx(x0[u].x), from_fx(x0[u].y), from_fx(x1[u].x), from_fx(x1[u].y))
                                : xf[u];
            if (live && ((ssq_mask >> kb[u]) & 1u)) {  // warp-uniform
                float q = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
#pragma unroll
                for (int o = 16; o; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
                if (c4 == 0) __stcg(c.m->ssq + (which * MK_MAXKB + kb[u]) * MK_MAXT + t, q);
            }
            const uint32_t w0 = pack_f16(v.x * g[u].x, v.y * g[u].y), w1 = pack_f16(v.z * g[u].z, v.w * g[u].w);
            bad |= f16x2_bad(w0) | f16x2_bad(w1);
            *reinterpret_cast<uint2 *>(fr + o_tc + kb[u] * 2048) = make_uint2(w0, w1);
        }
    }
    if (bad) range_err(300 + which);
}
// f32 activations [MK_MAXT][K] for the FFMA path
__device__ __noinline__ void build_act32(const ActSrc a, int K) {
    const Ctx c = make_ctx();
    float4 *dst = reinterpret_cast<float4 *>(c.sm + SM_SCRATCH);
    const int n4 = MK_MAXT * K / 4;
    for (int i0 = c.tid; i0 < n4; i0 += 4 * MK_NCWARPS * 32) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            int i = i0 + u * MK_NCWARPS * 32;
            int t = (4 * i) / K, col = 4 * i - t * K;
            v[u] = (i < n4 && t < c.T) ? act4(a, t, col) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            int i = i0 + u * MK_NCWARPS * 32;
            if (i < n4) dst[i] = v[u];
        }
    }
}

// k-blocks of a contiguous item range [b, e) over (.., rg, kc) ordered items
__device__ uint32_t needed_kb(int b, int e, const DMat &d) {
    if (e - b >= d.n_kc) return 0xffffffffu >> (32 - (d.cols / 128));
    // a chunk of cpk columns covers max(1, cpk / 128) blocks from block kc * cpk / 128
    const uint32_t span = d.cpk > 128 ? (1u << (d.cpk / 128)) - 1u : 1u;
    uint32_t mask = 0;
    for (int i = b; i < e; ++i) {
        int kc = i % d.n_kc;
        mask |= span << ((kc * d.cpk) / 128);
    }
    return mask;
}

// this CTA's input blocks of the fragment builds, for the launch (one thread)
__device__ __noinline__ void launch_masks() {
    const Ctx c = make_ctx();
    const DModel &m = *c.m;
    const DLayer &L = c.misc->L[0];
    uint32_t *k = c.misc->kbm;
    int b, e;
    split_range(L.qkv.n_rg * L.qkv.n_kc, c.G, c.cta, b, e);
    // the owners of the first row group's tiles cover every block once: they
    // also store the blocks' sum-of-squares partials
    const int nkc = L.qkv.n_kc;
    k[KBM_QKV] = needed_kb(b, e, L.qkv);
    k[KBM_QKV_SSQ] = b < nkc ? needed_kb(b, min(e, nkc), L.qkv) : 0u;
    split_range(L.o.n_rg * L.o.n_kc, c.G, c.cta, b, e);
    k[KBM_O] = needed_kb(b, e, L.o);
    k[KBM_RT] = chunk_kb_mask(c, m.H);
    k[KBM_RT_SSQ] = ssq_owner_mask(c, m.H);
}

// ------------------------------------------------------------------ GEMV tiles
// where the partial sums of one item go: token t's row r adds w * value into
// base[off(t) + r], with off(t) < 0 meaning token t does not take part
struct Tgt {
    long long *base;
    int st, tstride, ex, K2I, row_limit;
    const RouteSm *rt;
};
__device__ __forceinline__ Tgt make_tgt(const Ctx &c, int st, int ex, int mat, int rows, const RouteSm *rt) {
    const DModel &m = *c.m;
    Tgt g;
    g.st = st;
    g.ex = ex;
    g.rt = rt;
    g.row_limit = rows;
    g.K2I = m.K * 2 * m.I;
    switch (st) {
        case ST_QKV: g.base = acc_ptr(m, ACC_QKV, c.misc->par); g.tstride = m.nqkv; break;
        case ST_O: g.base = m.res; g.tstride = m.H; break;
        case ST_ROUTER: g.base = acc_ptr(m, ACC_RLOG, c.misc->par); g.tstride = m.E; break;
        case ST_SHA: g.base = acc_ptr(m, ACC_SH, c.misc->par) + mat * m.I; g.tstride = 2 * m.I; break;
        case ST_EXPA: g.base = acc_ptr(m, ACC_EA, c.misc->par) + mat * m.I; g.tstride = 2 * m.I; break;
        case ST_EXPB: g.base = m.res; g.tstride = m.H; break;
        default: g.base = m.logit_acc; g.tstride = m.V; break;
    }
    return g;
}
// offset of token t (< 0: not routed) and its weight
__device__ __forceinline__ int tgt_off(const Tgt &g, int t, int T, float &w) {
    w = 1.f;
    if (t >= T) return -1;
    if (g.st == ST_EXPA) {
        int j = g.rt->dslot[g.ex][t];
        return j < 0 ? -1 : t * g.K2I + j * g.tstride;
    }
    if (g.st == ST_EXPB && g.ex < g.rt->nd) {
        int j = g.rt->dslot[g.ex][t];
        if (j < 0) return -1;
        w = g.rt->w[t][j];
    }
    return t * g.tstride;
}

// MMA layout: for m-tile mt (0, 1) of the warp's 32 rows, lane holds rows
// (16mt + r, 16mt + r + 8) x tokens (2q, 2q+1) in acc[4mt .. 4mt+3]
__device__ __forceinline__ void flush_mma(const Ctx &c, const Tgt &g, int row0, const float *acc) {
    const int r = c.lane >> 2, q = c.lane & 3;
    float w0, w1;
    const int o0 = tgt_off(g, 2 * q, c.T, w0), o1 = tgt_off(g, 2 * q + 1, c.T, w1);
    uint32_t bad = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int o = (i & 1) ? o1 : o0;
        const float w = (i & 1) ? w1 : w0;
        const int row = row0 + (i >> 2) * 16 + r + ((i >> 1) & 1) * 8;
        if (o >= 0 && row < g.row_limit) {
            const float v = acc[i] * w;
            bad |= fx_bad(v);
            red_add(g.base + o + row, to_fx(v));
        }
    }
    if (bad) range_err(320 + g.st);
}
// FFMA layout: lane l holds row l of the warp's 32 rows, all tokens
__device__ __forceinline__ void flush_f32(const Ctx &c, const Tgt &g, int row0, const float *acc) {
    int row = row0 + c.lane;
    if (row >= g.row_limit) return;
    uint32_t bad = 0;
#pragma unroll
    for (int t = 0; t < MK_MAXT; ++t) {
        float w;
        const int o = tgt_off(g, t, c.T, w);
        if (o >= 0) {
            const float v = acc[t] * w;
            bad |= fx_bad(v);
            red_add(g.base + o + row, to_fx(v));
        }
    }
    if (bad) range_err(320 + g.st);
}

// one 256-row x 128-byte tile of FP8 or bf16 weights against the f16 fragments;
// warp w reduces rows 32w..32w+31 as two 16-row MMA tiles
__device__ __forceinline__ void tile_mma(const Ctx &c, int dtype, int slot, int kc, float *acc) {
    const int r = c.lane >> 2, q = c.lane & 3;
    const uint32_t tile = sa(c.sm + SM_RING + slot * MK_SLOT);
    const int rw = c.warp * 32 + r;  // rows rw, rw+8 (tile 0), rw+16, rw+24 (tile 1); all = r mod 8
    const uint32_t frag = sa(c.sm + SM_SCRATCH);
    if (dtype == MK_DT_FP8E4M3_B128) {
        const int ca = ((2 * q + (q >> 1)) ^ r) << 4, cb = ((2 * q + 1 - (q >> 1)) ^ r) << 4;
        uint4 a[4][2];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            a[j][0] = lds128(tile + (rw + 8 * j) * 128 + ca);
            a[j][1] = lds128(tile + (rw + 8 * j) * 128 + cb);
        }
        const uint32_t fb = frag + kc * 2048 + c.lane * 16;
        uint4 f0 = lds128(fb), f1 = lds128(fb + 512), f2 = lds128(fb + 1024), f3 = lds128(fb + 1536);
        const uint32_t fx[8] = {f0.x, f0.z, f1.x, f1.z, f2.x, f2.z, f3.x, f3.z};
        const uint32_t fy[8] = {f0.y, f0.w, f1.y, f1.w, f2.y, f2.w, f3.y, f3.w};
        float k[4][4];  // [tile*2 + chain][4]
#pragma unroll
        for (int i = 0; i < 4; ++i) k[i][0] = k[i][1] = k[i][2] = k[i][3] = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2) {
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const uint4 &u0 = a[2 * mt][s2 >> 2], &u8 = a[2 * mt + 1][s2 >> 2];
                const uint32_t w0 = (s2 & 3) == 0 ? u0.x : (s2 & 3) == 1 ? u0.y : (s2 & 3) == 2 ? u0.z : u0.w;
                const uint32_t w8 = (s2 & 3) == 0 ? u8.x : (s2 & 3) == 1 ? u8.y : (s2 & 3) == 2 ? u8.z : u8.w;
                uint32_t lo0, hi0, lo8, hi8;
                e4m3x4_f16(w0, lo0, hi0);
                e4m3x4_f16(w8, lo8, hi8);
                mma_f16(k[2 * mt + (s2 & 1)], lo0, lo8, hi0, hi8, fx[s2], fy[s2]);
            }
        }
        const float *sc = reinterpret_cast<const float *>(c.sm + SM_SCALE + slot * MK_SCALE_SLOT);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            const float s0 = sc[rw + 16 * mt], s8 = sc[rw + 16 * mt + 8];
            acc[4 * mt + 0] += (k[2 * mt][0] + k[2 * mt + 1][0]) * s0;
            acc[4 * mt + 1] += (k[2 * mt][1] + k[2 * mt + 1][1]) * s0;
            acc[4 * mt + 2] += (k[2 * mt][2] + k[2 * mt + 1][2]) * s8;
            acc[4 * mt + 3] += (k[2 * mt][3] + k[2 * mt + 1][3]) * s8;
        }
    } else if (!kF32 && dtype == MK_DT_MXFP4_B32) {
        // 256 rows x 256 columns: a 128-byte row holds activation blocks 2kc
        // and 2kc+1.  Lane q takes 16-byte chunk q of each block, i.e. columns
        // 32q .. 32q+31, the columns frag_col gives it; in step s it uses the
        // four codes of word ((s>>1) + 2(q>>1)) & 3, half s & 1.  A 32-column
        // group has one E8M0 scale, so the four lanes of an MMA step hold four
        // different scales: each lane multiplies its decoded weights by
        // 2^(e_q - e_max) in f16 (a power of two, exact unless below 2^-24),
        // and the block's partial sums take 2^(e_max - 127) afterwards, e_max
        // being the largest of the row's four group exponents in the block.
        const unsigned char *sc = c.sm + SM_SCALE + slot * MK_SCALE_SLOT;  // [8 groups][256 rows]
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int kb = 2 * kc + b;
            const int ch = ((4 * b + q) ^ r) << 4;
            uint4 a[4];
            uint32_t fac[4];
            float sx[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                a[j] = lds128(tile + (rw + 8 * j) * 128 + ch);
                // word w of the chunk serves steps 2w' and 2w'+1 with w = (w' + 2(q>>1)) & 3:
                // rotate once so that word w' sits at index w'
                if (q & 2) a[j] = make_uint4(a[j].z, a[j].w, a[j].x, a[j].y);
                const int e = sc[(4 * b + q) * 256 + rw + 8 * j];
                int em = max(e, __shfl_xor_sync(0xffffffffu, e, 1));
                em = max(em, __shfl_xor_sync(0xffffffffu, em, 2));
                fac[j] = pow2_f16x2(e - em);
                sx[j] = e8m0_f(em);
            }
            const uint32_t fb = frag + kb * 2048 + c.lane * 16;
            uint4 f0 = lds128(fb), f1 = lds128(fb + 512), f2 = lds128(fb + 1024), f3 = lds128(fb + 1536);
            const uint32_t fx[8] = {f0.x, f0.z, f1.x, f1.z, f2.x, f2.z, f3.x, f3.z};
            const uint32_t fy[8] = {f0.y, f0.w, f1.y, f1.w, f2.y, f2.w, f3.y, f3.w};
            float k[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) k[i][0] = k[i][1] = k[i][2] = k[i][3] = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const uint4 &u0 = a[2 * mt], &u8 = a[2 * mt + 1];
                    const uint32_t w0 = w == 0 ? u0.x : w == 1 ? u0.y : w == 2 ? u0.z : u0.w;
                    const uint32_t w8 = w == 0 ? u8.x : w == 1 ? u8.y : w == 2 ? u8.z : u8.w;
                    uint32_t p0[4], p8[4];
                    e2m1x8_f16(w0, p0[0], p0[1], p0[2], p0[3]);
                    e2m1x8_f16(w8, p8[0], p8[1], p8[2], p8[3]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        p0[i] = hmul2u(p0[i], fac[2 * mt]);
                        p8[i] = hmul2u(p8[i], fac[2 * mt + 1]);
                    }
                    // steps 2w (bytes 0, 1) and 2w + 1 (bytes 2, 3)
                    mma_f16(k[2 * mt], p0[0], p8[0], p0[1], p8[1], fx[2 * w], fy[2 * w]);
                    mma_f16(k[2 * mt + 1], p0[2], p8[2], p0[3], p8[3], fx[2 * w + 1], fy[2 * w + 1]);
                }
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const float s0 = sx[2 * mt], s8 = sx[2 * mt + 1];
                acc[4 * mt + 0] += (k[2 * mt][0] + k[2 * mt + 1][0]) * s0;
                acc[4 * mt + 1] += (k[2 * mt][1] + k[2 * mt + 1][1]) * s0;
                acc[4 * mt + 2] += (k[2 * mt][2] + k[2 * mt + 1][2]) * s8;
                acc[4 * mt + 3] += (k[2 * mt][3] + k[2 * mt + 1][3]) * s8;
            }
        }
    } else {  // bf16: the tile is half of a 128-column block
        const int h = kc & 1, kb = kc >> 1;
        const bool act = (q >> 1) == h;
        const int qq = q & 1;
        const uint32_t fb = frag + kb * 2048 + c.lane * 16;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int ch = ((4 * qq + ((i + 2 * h) & 3)) ^ r) << 4;
            uint4 ra[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                ra[j] = act ? lds128(tile + (rw + 8 * j) * 128 + ch) : make_uint4(0, 0, 0, 0);
            uint4 f = lds128(fb + i * 512);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const uint4 &x0 = ra[2 * mt], &x8 = ra[2 * mt + 1];
                mma_f16(acc + 4 * mt, bf16x2_f16x2(x0.x), bf16x2_f16x2(x8.x), bf16x2_f16x2(x0.y),
                        bf16x2_f16x2(x8.y), f.x, f.y);
                mma_f16(acc + 4 * mt, bf16x2_f16x2(x0.z), bf16x2_f16x2(x8.z), bf16x2_f16x2(x0.w),
                        bf16x2_f16x2(x8.w), f.z, f.w);
            }
        }
    }
}

// one 256-row x 32-column fp32 tile with FFMA (tiny fp32 models): lane l of
// warp w owns row 32w + l
__device__ __forceinline__ void tile_f32(const Ctx &c, int K, int slot, int kc, float *acc) {
    const uint32_t tile = sa(c.sm + SM_RING + slot * MK_SLOT);
    const float *act = reinterpret_cast<const float *>(c.sm + SM_SCRATCH);
    const int row = c.warp * 32 + c.lane;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint4 w = lds128(tile + row * 128 + ((i ^ (row & 7)) << 4));
        float wv[4] = {__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                       __uint_as_float(w.w)};
        int col = kc * 32 + 4 * i;
#pragma unroll
        for (int t = 0; t < MK_MAXT; ++t) {
            if (t < c.T) {
                const float *x = act + t * K + col;
                acc[t] += wv[0] * x[0] + wv[1] * x[1] + wv[2] * x[2] + wv[3] * x[3];
            }
        }
    }
}

// h_e = silu(a/rms) * (b/rms) fragments of one expert (or the shared one)
__device__ __forceinline__ float silu_mul(float a, float b) { return __fdividef(a, 1.f + __expf(-a)) * b; }

// expert intermediate h = silu(a/rms) * (b/rms) of one routed expert (or the
// shared one) as f16 fragments; eight blocks of loads are issued at once
__device__ __noinline__ void build_h_frags(const RouteSm *rt, int ex, bool f32path_) {
    constexpr bool f32path = kF32;
    (void)f32path_;
    const Ctx c = make_ctx();
    const DModel &m = *c.m;
    const bool shared = ex >= rt->nd;
    auto base = [&](int t) -> const long long * {
        if (t >= c.T) return nullptr;
        if (shared) return acc_ptr(m, ACC_SH, c.misc->par) + (long long)t * 2 * m.I;
        int j = rt->dslot[ex][t];
        return j < 0 ? nullptr : acc_ptr(m, ACC_EA, c.misc->par) + (long long)(t * m.K + j) * 2 * m.I;
    };
    if (f32path) {
        float *dst = reinterpret_cast<float *>(c.sm + SM_SCRATCH);
        for (int i = c.tid; i < MK_MAXT * m.I; i += MK_NCWARPS * 32) {
            int t = i / m.I, col = i - t * m.I;
            const long long *pa = base(t);
            float inv = t < c.T ? c.misc->inv_rms[1][t] : 0.f;
            dst[i] = pa ? silu_mul(from_fx(__ldcg(pa + col)) * inv, from_fx(__ldcg(pa + m.I + col)) * inv) : 0.f;
        }
        return;
    }
    // thread (t, c4) converts columns 4*c4 .. 4*c4+3 of token t in every
    // 128-column block: each warp reads one accumulator row as whole L2 lines
    const int t = c.tid >> 5, c4 = c.lane;
    const long long *pa = base(t);
    const float inv = t < c.T ? c.misc->inv_rms[1][t] : 0.f;
    unsigned char *fr = c.sm + SM_SCRATCH + frag_off(0, t, c4);
    const int nkb = m.I / 128;
    constexpr int B = 4;
    uint32_t bad = 0;
    for (int kb0 = 0; kb0 < nkb; kb0 += B) {
        longlong2 av[B][2], bv[B][2];
#pragma unroll
        for (int u = 0; u < B; ++u) {
            av[u][0] = av[u][1] = bv[u][0] = bv[u][1] = make_longlong2(0, 0);
            if (pa && kb0 + u < nkb) {
                const longlong2 *pp = reinterpret_cast<const longlong2 *>(pa + (kb0 + u) * 128 + 4 * c4);
                const longlong2 *pb = reinterpret_cast<const longlong2 *>(pa + m.I + (kb0 + u) * 128 + 4 * c4);
                av[u][0] = __ldcg(pp);
                av[u][1] = __ldcg(pp + 1);
                bv[u][0] = __ldcg(pb);
                bv[u][1] = __ldcg(pb + 1);
            }
        }
#pragma unroll
        for (int u = 0; u < B; ++u) {
            if (kb0 + u >= nkb) break;
            float h[4] = {0.f, 0.f, 0.f, 0.f};
            if (pa) {
                h[0] = silu_mul(from_fx(av[u][0].x) * inv, from_fx(bv[u][0].x) * inv);
                h[1] = silu_mul(from_fx(av[u][0].y) * inv, from_fx(bv[u][0].y) * inv);
                h[2] = silu_mul(from_fx(av[u][1].x) * inv, from_fx(bv[u][1].x) * inv);
                h[3] = silu_mul(from_fx(av[u][1].y) * inv, from_fx(bv[u][1].y) * inv);
            }
            const uint32_t w0 = pack_f16(h[0], h[1]), w1 = pack_f16(h[2], h[3]);
            bad |= f16x2_bad(w0) | f16x2_bad(w1);
            *reinterpret_cast<uint2 *>(fr + (kb0 + u) * 2048) = make_uint2(w0, w1);
        }
    }
    if (bad) range_err(310);
}


// consume this CTA's tiles of one GEMV stage
__device__ __forceinline__ void flush_item(const Ctx &c, int st, int ex, int mat, int rg, const MatR &d,
                                           const RouteSm *rt, const float *acc) {
    const Tgt g = make_tgt(c, st, ex, mat, d.rows, rt);
    if (kF32 && d.dtype == MK_DT_F32) flush_f32(c, g, rg * 256 + c.warp * 32, acc);
    else flush_mma(c, g, rg * 256 + c.warp * 32, acc);
}
// consume this CTA's tiles of one GEMV stage
__device__ __noinline__ uint32_t cons_gemv(int st, const DLayer *Lp, const RouteSm *rt, uint32_t ci) {
    const Ctx c = make_ctx();
    const DLayer &L = *Lp;
    StageIter it;
    stage_iter(it, c, st, L, rt);
    uint64_t *const full = c.full, *const empty = c.empty;
    const int lane = c.lane;
    float acc[MK_MAXT];
#pragma unroll
    for (int i = 0; i < MK_MAXT; ++i) acc[i] = 0.f;
    int cex = -1, cmat = 0, crg = 0, last_hex = -1;
    const bool prof = c.p->marks != nullptr;
    unsigned long long cy_wait = 0, cy_comp = 0, cy_other = 0, cy0 = prof ? clock64() : 0;
    const int ntiles = it.n;
    for (int k = 0; it.n > 0; --it.n, it.advance(), ++k) {
        const MatR &d = it.cur();
        if (k == 0 || it.item_start()) {  // a new (expert slot, matrix, row group) item starts
            if (k > 0) {
                flush_item(c, st, cex, cmat, crg, cmat || (st == ST_EXPB && cex >= it.nd) ? it.m1 : it.m0, rt, acc);
#pragma unroll
                for (int i = 0; i < MK_MAXT; ++i) acc[i] = 0.f;
            }
            cex = it.ex;
            cmat = it.mat;
            crg = it.rg;
            if (st == ST_EXPB && it.ex != last_hex) {
                // the first build needs no barrier before it: the grid barrier
                // that opened the stage already follows every warp's last use
                // of the fragment area
                if (k > 0) bar_consumers();
                build_h_frags(rt, it.ex, kF32);
                bar_consumers();
                last_hex = it.ex;
            }
        }
        const int slot = ci % MK_RING;
        if (k == 0) mark(c, st * 16 + 7);
        unsigned long long cy1 = prof ? clock64() : 0;
        if (mbar_wait(&full[slot], (ci / MK_RING) & 1, c, 200 + st)) {
            unsigned long long cy2 = prof ? clock64() : 0;
            if (k == 0) mark(c, st * 16 + 1);
            if (kF32 && d.dtype == MK_DT_F32) tile_f32(c, d.cols, slot, it.kc, acc);
            else tile_mma(c, d.dtype, slot, it.kc, acc);
            if (prof) {
                unsigned long long cy3 = clock64();
                cy_wait += cy2 - cy1;
                cy_comp += cy3 - cy2;
                cy_other += cy1 - cy0;
                cy0 = cy3;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        ++ci;
    }
    if (ntiles > 0)
        flush_item(c, st, cex, cmat, crg, cmat || (st == ST_EXPB && cex >= it.nd) ? it.m1 : it.m0, rt, acc);
    if (prof && c.lane == 0 && c.warp == 0) {
        mark_val(c, MK_MARKS - 64 + st * 4 + 0, 900 + st * 4 + 0, cy_wait);
        mark_val(c, MK_MARKS - 64 + st * 4 + 1, 900 + st * 4 + 1, cy_comp);
        mark_val(c, MK_MARKS - 64 + st * 4 + 2, 900 + st * 4 + 2, cy_other);
    }
    mark(c, st * 16 + 2);
    return ci;
}


// ------------------------------------------------------------------ small helpers
__device__ __noinline__ void zero_slice_nc(long long *p, long long n) {
    const Ctx c = make_ctx();
    int b, e;
    split_range((int)n, c.G, c.cta, b, e);
    for (int i = b + c.tid; i < e; i += MK_NCWARPS * 32) __stcg(p + i, 0ll);
}
// this CTA's share of clearing the accumulators of parity par
__device__ __noinline__ void zero_accs(int par) {
    const Ctx c = make_ctx();
    for (int w = ACC_QKV; w <= ACC_RLOG; ++w) zero_slice_nc(acc_ptr(*c.m, w, par), acc_elems(*c.m, w));
}
__device__ __forceinline__ void zero_slice(const Ctx &c, long long *p, long long n) {
    (void)c;
    zero_slice_nc(p, n);
}
// sum of squares of 128-column block kb = (this CTA's index) of the residual
// for every token, for the final norm and the all-fp32 build; elsewhere the
// partials are formed in build_frags
__device__ __noinline__ void ssq_block_nc(int which) {
    const Ctx c = make_ctx();
    const DModel &m = *c.m;
    int kb = c.cta;
    if (kb >= m.H / 128) return;
    if (c.warp >= c.T) return;
    int t = c.warp;
    float s = 0.f;
    for (int i = c.lane; i < 128; i += 32) {
        float v = from_fx(__ldcg(m.res + (long long)t * m.H + kb * 128 + i));
        s += v * v;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (c.lane == 0) __stcg(m.ssq + (which * MK_MAXKB + kb) * MK_MAXT + t, s);
}
__device__ __forceinline__ void ssq_block(const Ctx &c, int which) {
    (void)c;
    ssq_block_nc(which);
}
__device__ __noinline__ void compute_inv_rms_nc(int which) {
    const Ctx c = make_ctx();
    const DModel &m = *c.m;
    if (c.warp < c.T) {
        const int t = c.warp;
        float v = c.lane < m.H / 128 ? __ldcg(m.ssq + (which * MK_MAXKB + c.lane) * MK_MAXT + t) : 0.f;
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (c.lane == 0) c.misc->inv_rms[which][t] = rsqrtf(v / (float)m.H + m.eps);
    }
}
__device__ __forceinline__ void compute_inv_rms(const Ctx &c, int which) {
    (void)c;
    compute_inv_rms_nc(which);
}

// ------------------------------------------------------------------ routing
// Selection key of expert e: the order-preserving bit pattern of s + b with
// its 9 lowest significand bits replaced by 511 - e, so that larger keys win
// and, between keys within 2^-14 relative of each other, the lower expert
// index wins.  (Routing is compared exactly only where the 8th and 9th keys
// differ by more than 1e-3.)
__device__ __forceinline__ uint32_t key32(float key, int e) {
    uint32_t b = __float_as_uint(key);
    b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return (b & ~0x1ffu) | (uint32_t)(511 - e);
}
// sort 16 keys descending (bitonic network, registers)
__device__ __forceinline__ void bitonic16_desc(uint32_t *v) {
#pragma unroll
    for (int k = 2; k <= 16; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                int l = i ^ j;
                if (l > i) {
                    const uint32_t a = v[i], b = v[l];
                    const bool desc = (i & k) == 0;
                    v[i] = desc ? max(a, b) : min(a, b);
                    v[l] = desc ? min(a, b) : max(a, b);
                }
            }
        }
    }
}

// Routing of the block, every CTA redundantly.  Warp t < T takes token t:
// one batch of loads brings its sum-of-squares partials (for the MoE RMSNorm)
// and its router logits; keys s + b (selection bias) are sorted 16 per lane
// by a bitonic network and merged across the warp to the top K; the weights
// are the unbiased scores of the chosen experts (taken from their owner lanes
// by shuffle) normalised to 1.  The distinct experts of the block and each
// (expert slot, token) pair then come from a bit mask and a prefix count.
__device__ __noinline__ void route_layer(const DLayer *Lp, RouteSm *rt) {
    const Ctx c = make_ctx();
    const DLayer &L = *Lp;
    const DModel &m = *c.m;
    mark(c, ST_EXPA * 16 + 4);
    if (c.tid < 16) c.misc->emask[c.tid] = 0;
    for (int i = c.tid; i < MK_MAXD * MK_MAXT / 4; i += MK_NCWARPS * 32)
        reinterpret_cast<int *>(&rt->dslot[0][0])[i] = -1;
    bar_consumers();
    if (c.warp < c.T) {
        const int t = c.warp;
        float sq = c.lane < m.H / 128 ? __ldcg(m.ssq + (MK_MAXKB + c.lane) * MK_MAXT + t) : 0.f;
        long long raw[16];
        float bias[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int e = c.lane + 32 * i;
            raw[i] = 0;
            bias[i] = 0.f;
            if (e < m.E) {
                raw[i] = __ldcg(acc_ptr(m, ACC_RLOG, c.misc->par) + (long long)t * m.E + e);
                bias[i] = __ldg(L.router_bias + e);
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        const float inv = rsqrtf(sq / (float)m.H + m.eps);
        if (c.lane == 0) c.misc->inv_rms[1][t] = inv;
        float sg[16];
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int e = c.lane + 32 * i;
            sg[i] = 0.f;  // register rows past the last expert hold no score
            if (32 * i < m.E) sg[i] = 1.f / (1.f + expf(-from_fx(raw[i]) * inv));
            v[i] = e < m.E ? key32(sg[i] + bias[i], e) : 0u;
        }
        bitonic16_desc(v);
        // bitonic merge of the lanes' sorted top-8 lists
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t pv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) pv[i] = __shfl_xor_sync(0xffffffffu, v[i], o);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = max(v[i], pv[7 - i]);
#pragma unroll
            for (int jj = 4; jj > 0; jj >>= 1) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if ((i & jj) == 0) {
                        const uint32_t a = v[i], b = v[i + jj];
                        v[i] = max(a, b);
                        v[i + jj] = min(a, b);
                    }
                }
            }
        }
        // lane j < K takes entry j of the merged list
        uint32_t mine = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i == c.lane) mine = v[i];
        const int e = 511 - (int)(mine & 0x1ffu);
        // the unbiased score of lane j's expert e: register e >> 5 of lane e & 31,
        // fetched with one shuffle per register index
        float s = 0.f;
        const int src = e & 31, hi = e >> 5;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float val = __shfl_sync(0xffffffffu, sg[i], src);
            if (i == hi) s = val;
        }
        float sum = c.lane < m.K ? s : 0.f;
#pragma unroll
        for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (c.lane < m.K) {
            rt->idx[t][c.lane] = e;
            rt->w[t][c.lane] = s / sum;
            atomicOr(&c.misc->emask[e >> 5], 1 << (e & 31));
        }
    }
    bar_consumers();
    mark(c, ST_EXPA * 16 + 6);
    if (c.warp == 0) {
        const int cnt = c.lane < 16 ? __popc(c.misc->emask[c.lane]) : 0;
        int pre = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, pre, o);
            if (c.lane >= o) pre += y;
        }
        if (c.lane < 16) {
            int pos = pre - cnt;
            c.misc->epre[c.lane] = pos;
            uint32_t w = c.misc->emask[c.lane];
            while (w) {
                rt->dlist[pos++] = c.lane * 32 + __ffs(w) - 1;
                w &= w - 1;
            }
        }
        if (c.lane == 31) rt->nd = pre;
    } else if (c.warp <= 2) {
        // meanwhile warps 1 and 2 work out this CTA's split of the routed
        // gate/up and down stages, which the producer and the consumers read
        const int nd = __reduce_add_sync(0xffffffffu, c.lane < 16 ? __popc(c.misc->emask[c.lane]) : 0);
        if (c.lane == 0) stage_seed(rt->seed[c.warp - 1], c, c.warp == 1 ? ST_EXPA : ST_EXPB, L, nd);
    }
    bar_consumers();
    if (c.warp < c.T && c.lane < m.K) {
        const int t = c.warp, e = rt->idx[t][c.lane], wd = e >> 5;
        const int pos = c.misc->epre[wd] + __popc(c.misc->emask[wd] & ((1u << (e & 31)) - 1u));
        rt->dslot[pos][t] = (signed char)c.lane;
    }
    bar_consumers();
}

// ------------------------------------------------------------------ attention
// q rows are ordered (t, head-in-group): row = t * G + hh
__device__ float qkv_val(const Ctx &c, int t, int col) {
    return from_fx(__ldcg(acc_ptr(*c.m, ACC_QKV, c.misc->par) + (long long)t * c.m->nqkv + col)) *
           c.misc->inv_rms[0][t];
}

// prepares rotated q (scratch) and, for the unit holding the new block, the
// block's K/V (scratch + cache append)
template <bool kFP8>
__device__ __forceinline__ void att_prepare(const Ctx &c, int l, const AttUnit &u, bool mma_path) {
    const DModel &m = *c.m;
    // head dim 128 on the tensor-core path, 64 in the all-fp32 build; rows
    // divide by G through its 16-bit reciprocal (exact for rows below 1024)
    constexpr int hd = kF32 ? 32 : 64;
    const int G = m.Hq / m.Hkv, R = G * c.T;
    const uint32_t ginv = (65536u + G - 1) / G;
    constexpr bool fp8kv = kFP8;
    bool qbad = false;
    unsigned char *scr = c.sm + SM_SCRATCH;
    const long long *qkv = acc_ptr(m, ACC_QKV, c.misc->par);
    // rotated queries: 4 consecutive pairs per item, two items per thread and batch
    constexpr int nk4 = hd / 4;
    const int nitem = R * nk4;
    longlong2 xa[2][2], xb[2][2];
    float4 ra[2][2];
    auto load = [&](int i0) {
#pragma unroll
        for (int u4 = 0; u4 < 2; ++u4) {
            int i = i0 + u4 * MK_NCWARPS * 32;
            if (i < nitem) {
                int row = i / nk4, k = (i - row * nk4) * 4;
                int t = (int)(((uint32_t)row * ginv) >> 16), h = u.g * G + (row - t * G);
                const long long *b = qkv + (long long)t * m.nqkv + h * m.d + k;
                xa[u4][0] = __ldcg(reinterpret_cast<const longlong2 *>(b));
                xa[u4][1] = __ldcg(reinterpret_cast<const longlong2 *>(b) + 1);
                xb[u4][0] = __ldcg(reinterpret_cast<const longlong2 *>(b + hd));
                xb[u4][1] = __ldcg(reinterpret_cast<const longlong2 *>(b + hd) + 1);
                const float4 *rp = reinterpret_cast<const float4 *>(m.rope + (long long)(c.ctx + t) * hd + k);
                ra[u4][0] = __ldg(rp);
                ra[u4][1] = __ldg(rp + 1);
            }
        }
    };
    // the first batch of query loads and the attention RMSNorm factors (warp t
    // reduces token t's 128-column sum-of-squares partials) are in flight together
    load(c.tid);
    if (c.warp < c.T) {
        const int t = c.warp;
        float v = c.lane < m.H / 128 ? __ldcg(m.ssq + c.lane * MK_MAXT + t) : 0.f;
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (c.lane == 0) c.misc->inv_rms[0][t] = rsqrtf(v / (float)m.H + m.eps);
    }
    bar_consumers();
    for (int i0 = c.tid; i0 < nitem; i0 += 2 * MK_NCWARPS * 32) {
        if (i0 != c.tid) load(i0);
#pragma unroll
        for (int u4 = 0; u4 < 2; ++u4) {
            int i = i0 + u4 * MK_NCWARPS * 32;
            if (i >= nitem) break;
            int row = i / nk4, k = (i - row * nk4) * 4;
            float inv = c.misc->inv_rms[0][((uint32_t)row * ginv) >> 16];
            float x1[4] = {from_fx(xa[u4][0].x), from_fx(xa[u4][0].y), from_fx(xa[u4][1].x), from_fx(xa[u4][1].y)};
            float x2[4] = {from_fx(xb[u4][0].x), from_fx(xb[u4][0].y), from_fx(xb[u4][1].x), from_fx(xb[u4][1].y)};
            float cs[8] = {ra[u4][0].x, ra[u4][0].y, ra[u4][0].z, ra[u4][0].w,
                           ra[u4][1].x, ra[u4][1].y, ra[u4][1].z, ra[u4][1].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float a1 = x1[j] * inv, a2 = x2[j] * inv;
                float y1 = a1 * cs[2 * j] - a2 * cs[2 * j + 1], y2 = a2 * cs[2 * j] + a1 * cs[2 * j + 1];
                if constexpr (fp8kv) {
                    __half *qs = reinterpret_cast<__half *>(scr);
                    const __half h1 = __float2half_rn(y1), h2 = __float2half_rn(y2);
                    qbad |= (__habs(h1) > __float2half_rn(65504.f)) | (__habs(h2) > __float2half_rn(65504.f)) |
                            __hisnan(h1) | __hisnan(h2);
                    qs[row * 136 + q_col_fp8(k + j)] = h1;
                    qs[row * 136 + q_col_fp8(k + j + hd)] = h2;
                } else if (mma_path) {
                    __nv_bfloat16 *qs = reinterpret_cast<__nv_bfloat16 *>(scr);
                    qs[row * 136 + k + j] = __float2bfloat16_rn(y1);
                    qs[row * 136 + k + j + hd] = __float2bfloat16_rn(y2);
                } else {
                    float *qs = reinterpret_cast<float *>(scr);
                    qs[row * m.d + k + j] = y1;
                    qs[row * m.d + k + j + hd] = y2;
                }
            }
        }
    }
    if (qbad) range_err(331);
    if (mma_path) {  // zero the padding rows of the last m-tile (zero bits in bf16 and f16)
        uint16_t *qs = reinterpret_cast<uint16_t *>(scr);
        int R16 = (R + 15) & ~15;
        for (int i = c.tid; i < (R16 - R) * 136; i += MK_NCWARPS * 32) qs[R * 136 + i] = 0;
    }
    if (!u.has_new) return;
    // block keys / values: mini page after the queries
    unsigned char *mini = scr + 17408;
    if (mma_path) {
        for (int i = c.tid; i < 8192 / 16; i += MK_NCWARPS * 32)
            reinterpret_cast<uint4 *>(mini)[i] = make_uint4(0, 0, 0, 0);
    }
    bar_consumers();
    const int kv_es = m.kv_es;
    for (int i = c.tid; i < c.T * hd; i += MK_NCWARPS * 32) {
        int t = i / hd, k = i - t * hd;
        int kc0 = (m.Hq + u.g) * m.d, vc0 = (m.Hq + m.Hkv + u.g) * m.d;
        float x1 = qkv_val(c, t, kc0 + k), x2 = qkv_val(c, t, kc0 + k + hd);
        float2 cs = __ldg(m.rope + (long long)(c.ctx + t) * hd + k);
        float k1 = x1 * cs.x - x2 * cs.y, k2 = x2 * cs.x + x1 * cs.y;
        float v1 = qkv_val(c, t, vc0 + k), v2 = qkv_val(c, t, vc0 + k + hd);
        int pos = c.ctx + t;
        int phys = __ldg(c.p->page_table + pos / m.P);
        long long off = ((long long)(phys * m.Hkv + u.g) * m.P + (pos % m.P)) * m.d;
        if constexpr (kFP8) {
            // codes of value / scale (nearest, ties to even, saturating at 448)
            const float ks = c.p->kv_scale[2 * l], vs = c.p->kv_scale[2 * l + 1];
            const unsigned char kc1 = e4m3_code(k1 / ks), kc2 = e4m3_code(k2 / ks);
            const unsigned char vc1 = e4m3_code(v1 / vs), vc2 = e4m3_code(v2 / vs);
            unsigned char *kp = reinterpret_cast<unsigned char *>(c.p->kpool[l]) + off;
            unsigned char *vp = reinterpret_cast<unsigned char *>(c.p->vpool[l]) + off;
            kp[k] = kc1;
            kp[k + hd] = kc2;
            vp[k] = vc1;
            vp[k + hd] = vc2;
            // mini page [16 keys][128 B] swizzled, as the pages of the ring
            auto put = [&](unsigned char *base, int dd, unsigned char v) { base[swz(0, t, dd)] = v; };
            put(mini, k, kc1);
            put(mini, k + hd, kc2);
            put(mini + 4096, k, vc1);
            put(mini + 4096, k + hd, vc2);
        } else if (kv_es == 2) {
            __nv_bfloat16 kb1 = __float2bfloat16_rn(k1), kb2 = __float2bfloat16_rn(k2);
            __nv_bfloat16 vb1 = __float2bfloat16_rn(v1), vb2 = __float2bfloat16_rn(v2);
            __nv_bfloat16 *kp = reinterpret_cast<__nv_bfloat16 *>(c.p->kpool[l]) + off;
            __nv_bfloat16 *vp = reinterpret_cast<__nv_bfloat16 *>(c.p->vpool[l]) + off;
            kp[k] = kb1;
            kp[k + hd] = kb2;
            vp[k] = vb1;
            vp[k + hd] = vb2;
            if (mma_path) {  // [box][16 keys][128 B] swizzled
                auto put = [&](unsigned char *base, int dd, __nv_bfloat16 v) {
                    int byte = dd * 2;
                    int bx = byte >> 7;
                    *reinterpret_cast<__nv_bfloat16 *>(base + (swz(0, t, byte & 127) + bx * 2048)) = v;
                };
                put(mini, k, kb1);
                put(mini, k + hd, kb2);
                put(mini + 4096, k, vb1);
                put(mini + 4096, k + hd, vb2);
            } else {
                float *mk = reinterpret_cast<float *>(mini);
                mk[t * m.d + k] = __bfloat162float(kb1);
                mk[t * m.d + k + hd] = __bfloat162float(kb2);
                mk[1024 + t * m.d + k] = __bfloat162float(vb1);
                mk[1024 + t * m.d + k + hd] = __bfloat162float(vb2);
            }
        } else {
            float *kp = reinterpret_cast<float *>(c.p->kpool[l]) + off;
            float *vp = reinterpret_cast<float *>(c.p->vpool[l]) + off;
            kp[k] = k1;
            kp[k + hd] = k2;
            vp[k] = v1;
            vp[k + hd] = v2;
            float *mk = reinterpret_cast<float *>(mini);
            mk[t * m.d + k] = k1;
            mk[t * m.d + k + hd] = k2;
            mk[1024 + t * m.d + k] = v1;
            mk[1024 + t * m.d + k + hd] = v2;
        }
    }
}

// tensor-core attention state of one warp (16 query rows, d = 128)
struct AttMma {
    uint32_t qaddr;       // ldmatrix row address of this lane in the rotated queries
    float o[16][4];
    float mrow[2], lrow[2];
};

// one key page of nkeys (64, or 16 for the block's own keys): kbase/vbase hold
// [2 boxes][nkeys][128 B] swizzled with box stride bs.  Keys are taken in
// 32-key halves, each with its own online-softmax update.
__device__ __forceinline__ void att_page_mma(const Ctx &c, AttMma &A, uint32_t kbase, uint32_t vbase, int bs,
                             int k0, int nkeys, int valid, bool causal, int mt, int G) {
    const int r = c.lane >> 2, q = c.lane & 3, mi = c.lane >> 3, li = c.lane & 7;
    const float sl2 = rsqrtf((float)c.m->d) * 1.4426950408889634f;
    for (int h0 = k0; h0 < nkeys; h0 += 32) {
        const int nnt = min(4, (nkeys - h0) >> 3);
        float sc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t q0, q1, q2, q3;  // query fragment of head dims 16kk..16kk+15
            ldsm4(A.qaddr + kk * 32, q0, q1, q2, q3);
#pragma unroll
            for (int pp = 0; pp < 2; ++pp) {
                if (2 * pp < nnt) {
                    int key = h0 + 8 * (2 * pp + (mi >> 1)) + li;
                    int dch = 2 * kk + (mi & 1);
                    uint32_t ad = kbase + (dch >> 3) * bs + key * 128 + (((dch & 7) ^ (key & 7)) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm4(ad, b0, b1, b2, b3);
                    mma_bf16(sc[2 * pp], q0, q1, q2, q3, b0, b1);
                    mma_bf16(sc[2 * pp + 1], q0, q1, q2, q3, b2, b3);
                }
            }
        }
        // mask, scale, online softmax (log2 domain)
        float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                int key = h0 + 8 * nt + 2 * q + (i & 1);
                int row = mt * 16 + r + (i >> 1) * 8;
                bool ok = nt < nnt && key < valid;
                if (causal) ok = ok && key <= row / G;
                float v = ok ? sc[nt][i] * sl2 : -CUDART_INF_F;
                sc[nt][i] = v;
                mx[i >> 1] = fmaxf(mx[i >> 1], v);
            }
        }
        float corr[2], mn[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
            mn[h] = fmaxf(A.mrow[h], mx[h]);
            corr[h] = exp2f(A.mrow[h] - mn[h]);
            A.mrow[h] = mn[h];
            A.lrow[h] *= corr[h];
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float pv = exp2f(sc[nt][i] - mn[i >> 1]);
                sc[nt][i] = pv;
                A.lrow[i >> 1] += pv;
            }
        }
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) {
            A.o[nd][0] *= corr[0];
            A.o[nd][1] *= corr[0];
            A.o[nd][2] *= corr[1];
            A.o[nd][3] *= corr[1];
        }
        // P V over the half's 16-key steps
        const bool partial = valid < h0 + 8 * nnt;
#pragma unroll
        for (int kk2 = 0; kk2 < 2; ++kk2) {
            if (2 * kk2 < nnt) {
                uint32_t a0 = pack_bf16(sc[2 * kk2][0], sc[2 * kk2][1]);
                uint32_t a1 = pack_bf16(sc[2 * kk2][2], sc[2 * kk2][3]);
                uint32_t a2 = pack_bf16(sc[2 * kk2 + 1][0], sc[2 * kk2 + 1][1]);
                uint32_t a3 = pack_bf16(sc[2 * kk2 + 1][2], sc[2 * kk2 + 1][3]);
                const int klo = h0 + 16 * kk2 + 2 * q;
                uint32_t m0 = 0xffffffffu, m1 = 0xffffffffu;
                if (partial) {
                    m0 = (klo < valid ? 0xffffu : 0u) | (klo + 1 < valid ? 0xffff0000u : 0u);
                    m1 = (klo + 8 < valid ? 0xffffu : 0u) | (klo + 9 < valid ? 0xffff0000u : 0u);
                }
#pragma unroll
                for (int np = 0; np < 8; ++np) {
                    int key = h0 + 16 * kk2 + li + (mi & 1) * 8;
                    int dch = 2 * np + (mi >> 1);
                    uint32_t ad = vbase + (dch >> 3) * bs + key * 128 + (((dch & 7) ^ (key & 7)) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm4t(ad, b0, b1, b2, b3);
                    mma_bf16(A.o[2 * np], a0, a1, a2, a3, b0 & m0, b1 & m1);
                    mma_bf16(A.o[2 * np + 1], a0, a1, a2, a3, b2 & m0, b3 & m1);
                }
            }
        }
    }
}

// one key page of FP8 E4M3 codes (nkeys 64, or 16 for the block's own keys):
// kbase / vbase hold [nkeys][128 B] swizzled.  Both products run as f16 MMAs on
// the codes, which f16 holds exactly; the K scale is part of sl2 (the softmax
// scale in the log2 domain) and the caller applies the V scale to the output.
// QK^T: head dims in the order of q_col_fp8, each lane reading two 16-byte
// chunks of its key row per 32-key half.  PV: output column n of n-tile
// 4g + np is physical head dim 32g + 4n + np, so a lane builds its B fragments
// from one 4-byte word (4 dims) of each of its four key rows.
__device__ __forceinline__ void att_page_fp8(const Ctx &c, AttMma &A, uint32_t kbase, uint32_t vbase, int k0, int nkeys,
                             int valid, bool causal, int mt, int G, float sl2) {
    const int r = c.lane >> 2, q = c.lane & 3;
    for (int h0 = k0; h0 < nkeys; h0 += 32) {
        const int nnt = min(4, (nkeys - h0) >> 3);
        float sc[4][4];
        uint4 kw[4][2];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
            kw[nt][0] = kw[nt][1] = make_uint4(0, 0, 0, 0);
            if (nt < nnt) {
                const int key = h0 + 8 * nt + r;
                const uint32_t row = kbase + key * 128;
                kw[nt][0] = lds128(row + (((2 * q) ^ (key & 7)) << 4));
                kw[nt][1] = lds128(row + (((2 * q + 1) ^ (key & 7)) << 4));
            }
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t q0, q1, q2, q3;
            ldsm4(A.qaddr + kk * 32, q0, q1, q2, q3);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                if (nt < nnt) {
                    const uint4 &u = kw[nt][kk >> 2];
                    const uint32_t w = (kk & 3) == 0 ? u.x : (kk & 3) == 1 ? u.y : (kk & 3) == 2 ? u.z : u.w;
                    uint32_t lo, hi;
                    e4m3x4_f16(w, lo, hi);
                    mma_f16(sc[nt], q0, q1, q2, q3, lo, hi);
                }
            }
        }
        float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                int key = h0 + 8 * nt + 2 * q + (i & 1);
                int row = mt * 16 + r + (i >> 1) * 8;
                bool ok = nt < nnt && key < valid;
                if (causal) ok = ok && key <= row / G;
                float v = ok ? sc[nt][i] * sl2 : -CUDART_INF_F;
                sc[nt][i] = v;
                mx[i >> 1] = fmaxf(mx[i >> 1], v);
            }
        }
        float corr[2], mn[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
            mn[h] = fmaxf(A.mrow[h], mx[h]);
            corr[h] = exp2f(A.mrow[h] - mn[h]);
            A.mrow[h] = mn[h];
            A.lrow[h] *= corr[h];
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float pv = exp2f(sc[nt][i] - mn[i >> 1]);
                sc[nt][i] = pv;
                A.lrow[i >> 1] += pv;
            }
        }
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) {
            A.o[nd][0] *= corr[0];
            A.o[nd][1] *= corr[0];
            A.o[nd][2] *= corr[1];
            A.o[nd][3] *= corr[1];
        }
#pragma unroll
        for (int kk2 = 0; kk2 < 2; ++kk2) {
            if (2 * kk2 < nnt) {
                const uint32_t a0 = pack_f16(sc[2 * kk2][0], sc[2 * kk2][1]);
                const uint32_t a1 = pack_f16(sc[2 * kk2][2], sc[2 * kk2][3]);
                const uint32_t a2 = pack_f16(sc[2 * kk2 + 1][0], sc[2 * kk2 + 1][1]);
                const uint32_t a3 = pack_f16(sc[2 * kk2 + 1][2], sc[2 * kk2 + 1][3]);
                // this lane's keys k, k+1 (b0) and k+8, k+9 (b1); keys at or past
                // `valid` may hold any bits (NaN codes included): read as zero
                const int k0 = h0 + 16 * kk2 + 2 * q;
                const int ks[4] = {k0, k0 + 1, k0 + 8, k0 + 9};
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    uint32_t v[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int key = ks[i];
                        const uint32_t ad = vbase + key * 128 + (((2 * g + (r >> 2)) ^ (key & 7)) << 4) + 4 * (r & 3);
                        v[i] = key < valid ? lds32(ad) : 0u;
                    }
                    uint32_t b0[4], b1[4];
                    e4m3x4_f16(prmt(v[0], v[1], 0x5140u), b0[0], b0[1]);
                    e4m3x4_f16(prmt(v[0], v[1], 0x7362u), b0[2], b0[3]);
                    e4m3x4_f16(prmt(v[2], v[3], 0x5140u), b1[0], b1[1]);
                    e4m3x4_f16(prmt(v[2], v[3], 0x7362u), b1[2], b1[3]);
#pragma unroll
                    for (int np = 0; np < 4; ++np) mma_f16(A.o[4 * g + np], a0, a1, a2, a3, b0[np], b1[np]);
                }
            }
        }
    }
}
// column (head dim) of output fragment element (n-tile nd, lane quad q, c = 0/1)
__device__ __forceinline__ int att_ocol(bool fp8kv, int nd, int q, int c) {
    return fp8kv ? 32 * (nd >> 2) + 8 * q + 4 * c + (nd & 3) : nd * 8 + 2 * q + c;
}

// FFMA attention of one page for <= 16 rows (fp32 caches, head_dim 64)
struct AttF {
    float o[16][2];
    float mrow[16], lrow[16];
};
__device__ void att_page_f32(const Ctx &c, AttF &A, const float *qs, int R, int G,
                             const unsigned char *kb, const unsigned char *vb, int bs, int es,
                             bool plain, int key0, int nkeys, int valid, bool causal) {
    const DModel &m = *c.m;
    const int nd = 2;  // head_dim 64
    const float sl2 = rsqrtf((float)m.d) * 1.4426950408889634f;
    for (int key = key0; key < key0 + nkeys; ++key) {
        if (key >= valid) break;
        float kv[2], vv[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            kv[i] = vv[i] = 0.f;
            if (i < nd) {
                int dd = c.lane + 32 * i;
                if (plain) {
                    kv[i] = reinterpret_cast<const float *>(kb)[key * m.d + dd];
                    vv[i] = reinterpret_cast<const float *>(vb)[key * m.d + dd];
                } else {
                    int byte = dd * es;
                    uint32_t off = (byte >> 7) * bs + (swz(0, key, byte & 127));
                    if (es == 4) {
                        kv[i] = *reinterpret_cast<const float *>(kb + off);
                        vv[i] = *reinterpret_cast<const float *>(vb + off);
                    } else {
                        kv[i] = bf16_to_f(*reinterpret_cast<const uint16_t *>(kb + off));
                        vv[i] = bf16_to_f(*reinterpret_cast<const uint16_t *>(vb + off));
                    }
                }
            }
        }
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            if (rr < R) {
                float s = 0.f;
#pragma unroll
                for (int i = 0; i < 2; ++i) s += qs[rr * m.d + c.lane + 32 * i] * kv[i];
#pragma unroll
                for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (causal && key > rr / G) continue;
                s *= sl2;
                float mn = fmaxf(A.mrow[rr], s);
                float corr = exp2f(A.mrow[rr] - mn), p = exp2f(s - mn);
                A.mrow[rr] = mn;
                A.lrow[rr] = A.lrow[rr] * corr + p;
#pragma unroll
                for (int i = 0; i < 2; ++i) A.o[rr][i] = A.o[rr][i] * corr + p * vv[i];
            }
        }
    }
}

// returns the ring position after this CTA's pages, or -1 if the step aborted
// (one instance per KV format on the tensor-core path: FP8 pages or bf16 pages)
template <bool kFP8>
__device__ __noinline__ long long cons_att(int l, uint32_t ci) {
    const Ctx c = make_ctx();
    const DModel &m = *c.m;
    const AttUnit u = att_unit(c);
    const int G = m.Hq / m.Hkv, R = G * c.T;
    constexpr bool mma_path = !kF32;
    const int bs = m.P * 128;
    const int D2 = m.d + 2;
    constexpr bool fp8kv = mma_path && kFP8;
    const float ksc = fp8kv ? c.p->kv_scale[2 * l] : 1.f, vsc = fp8kv ? c.p->kv_scale[2 * l + 1] : 1.f;
    const float sl2 = rsqrtf((float)m.d) * 1.4426950408889634f * ksc;
    if (u.active) att_prepare<fp8kv>(c, l, u, mma_path);
    bar_consumers();
    mark(c, ST_ATT * 16 + 0);
    unsigned char *scr = c.sm + SM_SCRATCH;
    float *part = m.att_part + (long long)(u.g * MK_MAXSPLIT + u.s) * MK_MAXROWS * D2;
    if (u.active && mma_path) {
        // m-tiles of this launch's rows; the warp streams per m-tile follow the
        // largest block the state takes, not this launch's T, so that a row's
        // pages are summed and merged in the same order whatever the block
        // size (batch invariance at long contexts, where a split holds
        // several pages)
        const int nmt = (R + 15) / 16, nws = MK_NCWARPS / max(nmt, (G * m.maxT + 15) / 16);
        const int mt = c.warp % nmt, ws = c.warp / nmt;
        const bool wact = c.warp < nmt * nws;
        AttMma A;
        A.mrow[0] = A.mrow[1] = -1e30f;
        A.lrow[0] = A.lrow[1] = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) A.o[i][0] = A.o[i][1] = A.o[i][2] = A.o[i][3] = 0.f;
        {
            int row = mt * 16 + (c.lane & 7) + ((c.lane >> 3) & 1) * 8;
            A.qaddr = sa(scr) + row * 272 + (c.lane >> 4) * 16;
        }
        // work units are 32-key halves of pages, dealt round-robin to the warp
        // streams: with one page per split both halves run side by side
        for (int j = u.p0; j < u.pc1; ++j) {
            const int ks = ci % MK_RING;
            bool ok = mbar_wait(&c.full[ks], (ci / MK_RING) & 1, c, 210);
            const int valid = min(m.P, c.ctx - j * m.P);
            for (int h = 0; h < 2; ++h) {
                if (ok && wact && ((j - u.p0) * 2 + h) % nws == ws && 32 * h < valid) {
                    const uint32_t kb = sa(c.sm + SM_RING + ks * MK_SLOT);
                    if constexpr (fp8kv) att_page_fp8(c, A, kb, kb + MK_SLOT / 2, 32 * h, 32 * h + 32, valid, false, mt, G, sl2);
                    else att_page_mma(c, A, kb, kb + MK_SLOT / 2, bs, 32 * h, 32 * h + 32, valid, false, mt, G);
                }
            }
            __syncwarp();
            if (c.lane == 0) mbar_arrive(&c.empty[ks]);
            ci += 1;
        }
        if (u.has_new && wact && ((u.pc1 - u.p0) * 2) % nws == ws) {
            uint32_t mini = sa(scr + 17408);
            if constexpr (fp8kv) att_page_fp8(c, A, mini, mini + 4096, 0, 16, c.T, true, mt, G, sl2);
            else att_page_mma(c, A, mini, mini + 4096, 2048, 0, 16, c.T, true, mt, G);
        }
        // finish row sums
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            A.lrow[h] += __shfl_xor_sync(0xffffffffu, A.lrow[h], 1);
            A.lrow[h] += __shfl_xor_sync(0xffffffffu, A.lrow[h], 2);
        }
        bar_consumers();
        // merge the warp streams of each m-tile through scratch
        const int r = c.lane >> 2, q = c.lane & 3;
        float *mrg = reinterpret_cast<float *>(scr);
        const int WS = 16 * 128 + 32;
        if (wact && ws > 0) {
            float *w = mrg + ((ws - 1) * nmt + mt) * WS;
#pragma unroll
            for (int nd = 0; nd < 16; ++nd) {
                const int c0 = att_ocol(fp8kv, nd, q, 0), c1 = att_ocol(fp8kv, nd, q, 1);
                w[r * 128 + c0] = A.o[nd][0];
                w[r * 128 + c1] = A.o[nd][1];
                w[(r + 8) * 128 + c0] = A.o[nd][2];
                w[(r + 8) * 128 + c1] = A.o[nd][3];
            }
            if (q == 0) {
                w[2048 + r] = A.mrow[0];
                w[2048 + r + 8] = A.mrow[1];
                w[2064 + r] = A.lrow[0];
                w[2064 + r + 8] = A.lrow[1];
            }
        }
        bar_consumers();
        if (wact && ws == 0) {
            for (int o2 = 1; o2 < nws; ++o2) {
                const float *w = mrg + ((o2 - 1) * nmt + mt) * WS;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    int rr = r + 8 * h;
                    float m2 = w[2048 + rr], l2 = w[2064 + rr];
                    float mn = fmaxf(A.mrow[h], m2);
                    float a = exp2f(A.mrow[h] - mn), b = exp2f(m2 - mn);
                    A.mrow[h] = mn;
                    A.lrow[h] = A.lrow[h] * a + l2 * b;
#pragma unroll
                    for (int nd = 0; nd < 16; ++nd) {
                        A.o[nd][2 * h] = A.o[nd][2 * h] * a + w[rr * 128 + att_ocol(fp8kv, nd, q, 0)] * b;
                        A.o[nd][2 * h + 1] = A.o[nd][2 * h + 1] * a + w[rr * 128 + att_ocol(fp8kv, nd, q, 1)] * b;
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                int row = mt * 16 + r + 8 * h;
                if (row < R) {
                    float *dst = part + row * D2;
                    if constexpr (fp8kv) {  // the V scale, and 8 consecutive dims 32g + 8q .. +7 per lane
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            float4 lo, hi;
                            lo.x = A.o[4 * g][2 * h] * vsc;
                            lo.y = A.o[4 * g + 1][2 * h] * vsc;
                            lo.z = A.o[4 * g + 2][2 * h] * vsc;
                            lo.w = A.o[4 * g + 3][2 * h] * vsc;
                            hi.x = A.o[4 * g][2 * h + 1] * vsc;
                            hi.y = A.o[4 * g + 1][2 * h + 1] * vsc;
                            hi.z = A.o[4 * g + 2][2 * h + 1] * vsc;
                            hi.w = A.o[4 * g + 3][2 * h + 1] * vsc;
                            __stcg(reinterpret_cast<float2 *>(dst + 32 * g + 8 * q), make_float2(lo.x, lo.y));
                            __stcg(reinterpret_cast<float2 *>(dst + 32 * g + 8 * q + 2), make_float2(lo.z, lo.w));
                            __stcg(reinterpret_cast<float2 *>(dst + 32 * g + 8 * q + 4), make_float2(hi.x, hi.y));
                            __stcg(reinterpret_cast<float2 *>(dst + 32 * g + 8 * q + 6), make_float2(hi.z, hi.w));
                        }
                    } else {
#pragma unroll
                        for (int nd = 0; nd < 16; ++nd)
                            __stcg(reinterpret_cast<float2 *>(dst + nd * 8 + 2 * q),
                                   make_float2(A.o[nd][2 * h], A.o[nd][2 * h + 1]));
                    }
                    if (q == 0) {
                        __stcg(dst + m.d, A.mrow[h]);
                        __stcg(dst + m.d + 1, A.lrow[h]);
                    }
                }
            }
        }
    } else if (u.active) {
        // FFMA path: all warps share every page, each warp takes 8 keys
        AttF A;
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            A.mrow[rr] = -1e30f;
            A.lrow[rr] = 0.f;
            A.o[rr][0] = A.o[rr][1] = 0.f;
        }
        const float *qs = reinterpret_cast<const float *>(scr);
        const int kpw = m.P / MK_NCWARPS;
        for (int j = u.p0; j < u.pc1; ++j) {
            const int ks = ci % MK_RING;
            bool ok = mbar_wait(&c.full[ks], (ci / MK_RING) & 1, c, 212);
            if (ok) {
                int valid = min(m.P, c.ctx - j * m.P);
                unsigned char *kb = c.sm + SM_RING + ks * MK_SLOT;
                att_page_f32(c, A, qs, R, G, kb, kb + MK_SLOT / 2, bs, m.kv_es, false, c.warp * kpw, kpw,
                             valid, false);
            }
            __syncwarp();
            if (c.lane == 0) mbar_arrive(&c.empty[ks]);
            ci += 1;
        }
        if (u.has_new && c.warp == 0) {
            const unsigned char *mini = scr + 17408;
            att_page_f32(c, A, qs, R, G, mini, mini + 4096, 0, 4, true, 0, c.T, c.T, true);
        }
        bar_consumers();
        float *mrg = reinterpret_cast<float *>(scr);
        const int WS = 16 * m.d + 32, MO = 16 * m.d;
        float *w = mrg + c.warp * WS;
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            if (rr < R) {
#pragma unroll
                for (int i = 0; i < 2; ++i) w[rr * m.d + c.lane + 32 * i] = A.o[rr][i];
                if (c.lane == 0) {
                    w[MO + rr] = A.mrow[rr];
                    w[MO + 16 + rr] = A.lrow[rr];
                }
            }
        }
        bar_consumers();
        for (int i = c.tid; i < R * m.d; i += MK_NCWARPS * 32) {
            int rr = i / m.d, dd = i - rr * m.d;
            float mn = -1e30f;
            for (int o2 = 0; o2 < MK_NCWARPS; ++o2) mn = fmaxf(mn, mrg[o2 * WS + MO + rr]);
            float acc = 0.f, lsum = 0.f;
            for (int o2 = 0; o2 < MK_NCWARPS; ++o2) {
                float a = exp2f(mrg[o2 * WS + MO + rr] - mn);
                acc += a * mrg[o2 * WS + rr * m.d + dd];
                lsum += a * mrg[o2 * WS + MO + 16 + rr];
            }
            float *dst = part + rr * D2;
            __stcg(dst + dd, acc);
            if (dd == 0) {
                __stcg(dst + m.d, mn);
                __stcg(dst + m.d + 1, lsum);
            }
        }
    }
    // group barrier among the splits of this kv head, then merge assigned rows
    bar_consumers();
    mark(c, ST_ATT * 16 + 1);
    if (!u.active) return ci;
    if (c.tid == 0) {
        bool ok = !aborted(c);
        arrive_release(m.att_cnt + l * m.Hkv + u.g);
        if (ok) ok = spin_ge_s32(m.att_cnt + l * m.Hkv + u.g, c.nsplit, c, 220);
        c.misc->gs_ok = ok;
    }
    bar_consumers();
    mark(c, ST_ATT * 16 + 2);
    if (!c.misc->gs_ok) return -1;
    int r0, r1;
    split_range(R, c.nsplit, u.s, r0, r1);
    const int nr = r1 - r0, ns = c.nsplit;
    const float *pbase = m.att_part + (long long)(u.g * MK_MAXSPLIT) * MK_MAXROWS * D2;
    // log-sum-exp merge of my rows: two adjacent lanes share a (row, column
    // pair) and take half of the splits each, so that one batch of loads in
    // flight covers up to 2 * 19 splits; each lane folds its half with the
    // running maximum, then the two halves are folded by one shuffle
    constexpr int hp = kF32 ? 32 : 64;  // column pairs of a head (dim 64 / 128)
    const uint32_t ginv = (65536u + G - 1) / G;
    const long long sstr = (long long)MK_MAXROWS * D2;
    for (int item = c.tid; item < nr * hp * 2; item += MK_NCWARPS * 32) {  // warp-uniform bound
        const int half = item & 1, grp = item >> 1;
        const int rr = grp / hp, dp = grp - rr * hp;
        const float *prow = pbase + (long long)(r0 + rr) * D2;
        int s0, s1;
        split_range(ns, 2, half, s0, s1);
        float M = -1e30f, lsum = 0.f;
        float2 acc = make_float2(0.f, 0.f);
        constexpr int CH = 19;
        for (int sp0 = s0; sp0 < s1; sp0 += CH) {
            float mv[CH], lv[CH];
            float2 av[CH];
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                mv[k] = -1e30f;
                lv[k] = 0.f;
                av[k] = make_float2(0.f, 0.f);
                if (sp0 + k < s1) {
                    const float *pp = prow + (long long)(sp0 + k) * sstr;
                    mv[k] = __ldcg(pp + m.d);
                    lv[k] = __ldcg(pp + m.d + 1);
                    av[k] = __ldcg(reinterpret_cast<const float2 *>(pp + 2 * dp));
                }
            }
            float cm = M;
#pragma unroll
            for (int k = 0; k < CH; ++k) cm = fmaxf(cm, mv[k]);
            const float sc = exp2f(M - cm);
            lsum *= sc;
            acc.x *= sc;
            acc.y *= sc;
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                const float w = exp2f(mv[k] - cm);
                lsum += w * lv[k];
                acc.x += w * av[k].x;
                acc.y += w * av[k].y;
            }
            M = cm;
        }
        const float Mo = __shfl_xor_sync(0xffffffffu, M, 1), lo = __shfl_xor_sync(0xffffffffu, lsum, 1);
        const float ox = __shfl_xor_sync(0xffffffffu, acc.x, 1), oy = __shfl_xor_sync(0xffffffffu, acc.y, 1);
        if (half == 0) {
            const float Mn = fmaxf(M, Mo), a = exp2f(M - Mn), b = exp2f(Mo - Mn);
            const float il = 1.f / (lsum * a + lo * b);
            const int row = r0 + rr, t = (int)(((uint32_t)row * ginv) >> 16), h = u.g * G + (row - t * G);
            __stcg(reinterpret_cast<float2 *>(m.o_buf + (long long)t * m.Hq * m.d + h * m.d + 2 * dp),
                   make_float2((acc.x * a + ox * b) * il, (acc.y * a + oy * b) * il));
        }
    }
    mark(c, ST_ATT * 16 + 3);
    return ci;
}

// ------------------------------------------------------------------ consumer
// copy one layer's descriptors into shared memory (consumer threads)
__device__ __noinline__ void copy_layer_nc(DLayer *dst, const DLayer *src) {
    const Ctx c = make_ctx();
    const int nw = (int)(sizeof(DLayer) / 4);
    for (int i = c.tid; i < nw; i += MK_NCWARPS * 32)
        reinterpret_cast<uint32_t *>(dst)[i] = __ldg(reinterpret_cast<const uint32_t *>(src) + i);
}
__device__ __forceinline__ void copy_layer(const Ctx &c, DLayer *dst, const DLayer *src) {
    (void)c;
    copy_layer_nc(dst, src);
}

// fold (m2, s2) into (m, s): s = s 2^(m - M) + s2 2^(m2 - M), M = max(m, m2);
// an empty side has m = -inf and s = 0
__device__ __forceinline__ void lse_fold(float &m, float &s, float m2, float s2) {
    const float M = fmaxf(m, m2);
    if (M == -CUDART_INF_F) return;
    s = (m == -CUDART_INF_F ? 0.f : s * exp2f(m - M)) + (m2 == -CUDART_INF_F ? 0.f : s2 * exp2f(m2 - M));
    m = M;
}

// Verification by sampling, after the per-CTA slice maxima and sums are in
// place (out of line, and like every out-of-line routine here it rebuilds the
// thread's context itself instead of taking the caller's by reference).  Every CTA combines the slices in the same fixed order, so all reach
// the same probabilities, accept count n and draw target; the CTA whose
// vocabulary slice holds the target scans it and writes the drawn token.
// Returns n (the caller's CTA 0 reports it).
__device__ __noinline__ int sample_verify_step() {
    const Ctx c = make_ctx();
    const DModel &m = *c.m;
    const Params &p = *c.p;
    const float kt = 1.4426950408889634f / p.temperature;
    float *rowm = reinterpret_cast<float *>(c.sm + SM_SCRATCH + 16384);  // [T] max (log2 domain)
    float *rowz = rowm + MK_MAXT;                                          // [T] sum of 2^(y - max)
    int *sh = reinterpret_cast<int *>(rowz + MK_MAXT);                     // n, owner, excluded token
    float *shf = reinterpret_cast<float *>(sh + 4);                        // slice base, target
    float *part = shf + 4;                                                 // [threads] scan partials
    if (c.warp < c.T) {  // warp t: row t over the CTAs' slices, lanes strided, then a fixed tree
        const int t = c.warp;
        float mx = -CUDART_INF_F, sm = 0.f;
        for (int k = c.lane; k < c.G; k += 32)
            lse_fold(mx, sm, __ldcg(m.cand_m + k * MK_MAXT + t), __ldcg(m.cand_s + k * MK_MAXT + t));
#pragma unroll
        for (int o = 16; o; o >>= 1) lse_fold(mx, sm, __shfl_xor_sync(0xffffffffu, mx, o),
                                              __shfl_xor_sync(0xffffffffu, sm, o));
        if (c.lane == 0) {
            rowm[t] = mx;
            rowz[t] = sm;
        }
    }
    bar_consumers();
    if (c.tid == 0) {
        int n = 0;
        for (int i = 1; i < c.T; ++i) {
            const int d = __ldg(p.tokens + i);
            const float pd = exp2f(__ldcg(p.out_logits + (long long)(i - 1) * m.V + d) * kt - rowm[i - 1]) / rowz[i - 1];
            if (__ldg(p.uniforms + i - 1) < pd) n = i;
            else break;
        }
        const int r = n, ex = n < c.T - 1 ? __ldg(p.tokens + n + 1) : -1;
        const float Mr = rowm[r];
        const float wex = ex >= 0 ? exp2f(__ldcg(p.out_logits + (long long)r * m.V + ex) * kt - Mr) : 0.f;
        const float target = __ldg(p.uniforms + c.T - 1) * (rowz[r] - wex);
        // the slice holding the target, by the slices' sums in CTA order
        float acc = 0.f, base = 0.f;
        int owner = -1, last = 0;
        for (int k = 0; k < c.G; ++k) {
            int b, e;
            split_range(m.V, c.G, k, b, e);
            const float mk = __ldcg(m.cand_m + k * MK_MAXT + r);
            float sk = mk == -CUDART_INF_F ? 0.f : __ldcg(m.cand_s + k * MK_MAXT + r) * exp2f(mk - Mr);
            if (ex >= b && ex < e) sk = fmaxf(sk - wex, 0.f);
            if (sk > 0.f) last = k;
            if (owner < 0 && acc + sk > target) {
                owner = k;
                base = acc;
            }
            acc += sk;
        }
        if (owner < 0) {  // the target at the very top (rounding): the last slice with weight
            owner = last;
            int b, e;
            split_range(m.V, c.G, last, b, e);
            const float mk = __ldcg(m.cand_m + last * MK_MAXT + r);
            float sk = __ldcg(m.cand_s + last * MK_MAXT + r) * exp2f(mk - Mr);
            if (ex >= b && ex < e) sk = fmaxf(sk - wex, 0.f);
            base = acc - sk;
        }
        sh[0] = n;
        sh[1] = owner;
        sh[2] = ex;
        shf[0] = base;
        shf[1] = target;
    }
    bar_consumers();
    const int n = sh[0];
    if (c.cta != sh[1]) return n;
    // the owner: contiguous runs of its slice per thread, partial sums in index
    // order, then the first run whose cumulative sum passes the target
    const int r = n, ex = sh[2];
    const float Mr = rowm[r], base = shf[0], target = shf[1];
    int b, e;
    split_range(m.V, c.G, c.cta, b, e);
    const int nth = MK_NCWARPS * 32, len = e - b, run = (len + nth - 1) / nth;
    const int x0 = b + c.tid * run, x1 = min(e, x0 + run);
    const float *lg = p.out_logits + (long long)r * m.V;
    float ps = 0.f;
    for (int x = x0; x < x1; ++x)
        if (x != ex) ps += exp2f(__ldcg(lg + x) * kt - Mr);
    part[c.tid] = ps;
    bar_consumers();
    if (c.tid == 0) {
        float cum = base;
        int tok = -1, lastx = -1;
        for (int j = 0; j < nth && tok < 0; ++j) {
            const int y0 = b + j * run, y1 = min(e, y0 + run);
            if (y0 >= y1) break;
            if (cum + part[j] > target) {
                for (int x = y0; x < y1; ++x) {
                    if (x == ex) continue;
                    const float w = exp2f(__ldcg(lg + x) * kt - Mr);
                    if (w > 0.f) lastx = x;
                    cum += w;
                    if (cum > target) {
                        tok = x;
                        break;
                    }
                }
                if (tok < 0) tok = lastx;  // rounding between the run's sum and its terms
            } else {
                cum += part[j];
                if (part[j] > 0.f) {
                    for (int x = y1 - 1; x >= y0; --x)
                        if (x != ex) {
                            lastx = x;
                            break;
                        }
                }
            }
        }
        if (tok < 0) tok = lastx >= 0 ? lastx : b;
        *p.out_token = tok;
    }
    return n;
}

__device__ __noinline__ void consumer() {
    const Ctx c = make_ctx();
    const DModel &m = *c.m;
    const Params &p = *c.p;
    uint32_t ci = 0;
    constexpr bool f32path = kF32;
    const uint32_t allH = 0xffffffffu >> (32 - m.H / 128);
    int nl = p.mode ? 1 : m.L;
    // zero the accumulators, load the residual stream
    // the first layer's accumulators (parity 0); each layer clears the next
    // layer's copy while it waits at the barrier that ends its QKV stage
    zero_accs(0);
    if (p.mode == 0) zero_slice(c, m.logit_acc, (long long)c.T * m.V);
    if (c.cta == 0) {
        for (int i = c.tid; i < m.L * m.Hkv; i += MK_NCWARPS * 32) __stcg(m.att_cnt + i, 0);
    }
    {
        long long n = (long long)c.T * m.H;
        long long b = n * c.cta / c.G, e = n * (c.cta + 1) / c.G;
        for (long long i = b + c.tid; i < e; i += MK_NCWARPS * 32) {
            int t = (int)(i / m.H), col = (int)(i - (long long)t * m.H);
            float v = p.mode ? __ldg(p.hidden_in + i)
                             : bf16_to_f(__ldg(m.embed + (long long)__ldg(p.tokens + t) * m.H + col));
            if (fx_bad(v)) range_err(330);
            __stcg(m.res + (long long)t * m.H + col, to_fx(v));
        }
    }
    if (!grid_sync(c, 1)) return;
    for (int li = 0; li < nl; ++li) {
        const int l = p.mode ? p.layer : li;
        const DLayer &L = c.misc->L[li & 1];
        RouteSm *rt = &c.rt[li & 1];
        if (c.tid == 0) c.misc->par = li & 1;  // read after the CTA barriers below
        // ---- QKV
        {
            mark(c, ST_QKV * 16 + 5);
            ActSrc a{m.res, nullptr, m.H, L.attn_norm};
            if (f32path) {
                build_act32(a, m.H);
                ssq_block(c, 0);
            } else {
                build_frags(a, c.misc->kbm[KBM_QKV], c.misc->kbm[KBM_QKV_SSQ], 0);
            }
            mark(c, ST_QKV * 16 + 6);
            bar_consumers();
            mark(c, ST_QKV * 16 + 0);
            ci = cons_gemv(ST_QKV, &(L), rt, ci);
            grid_arrive(c);
            // the next layer's accumulators: their copy was last read in the
            // previous layer, which every CTA has left
            zero_accs((li + 1) & 1);
            if (!grid_wait(c, 2)) return;
        }
        // ---- attention
        {
            const long long r = (!kF32 && m.kvdt == MK_DT_FP8E4M3) ? cons_att<true>(l, ci) : cons_att<false>(l, ci);
            if (r < 0) return;
            ci = (uint32_t)r;
        }
        if (!grid_sync(c, 3)) return;
        // ---- O projection (+ residual)
        {
            mark(c, ST_O * 16 + 5);
            ActSrc a{nullptr, m.o_buf, m.Hq * m.d, nullptr};
            if (f32path) build_act32(a, m.Hq * m.d);
            else build_frags(a, c.misc->kbm[KBM_O]);
            mark(c, ST_O * 16 + 6);
            bar_consumers();
            mark(c, ST_O * 16 + 0);
            ci = cons_gemv(ST_O, &(L), rt, ci);
            if (!grid_sync(c, 4)) return;
        }
        // ---- router + shared expert gate/up, then routed gate/up
        {
            ActSrc a{m.res, nullptr, m.H, L.moe_norm};
            mark(c, ST_ROUTER * 16 + 8);
            if (f32path) {
                build_act32(a, m.H);
                ssq_block(c, 1);
            } else {
                build_frags(a, c.misc->kbm[KBM_RT], c.misc->kbm[KBM_RT_SSQ], 1);
            }
            mark(c, ST_ROUTER * 16 + 6);
            bar_consumers();
            mark(c, ST_ROUTER * 16 + 0);
            ci = cons_gemv(ST_ROUTER, &(L), rt, ci);
            grid_arrive(c);
            ci = cons_gemv(ST_SHA, &(L), rt, ci);
            // descriptors of the next layer, copied while the barrier settles.
            // The producer reads them only after this layer's routing, which
            // these threads publish after the copy.
            if (p.mode == 0 && li + 1 < nl) copy_layer(c, &c.misc->L[(li + 1) & 1], m.layers + li + 1);
            if (!grid_wait(c, 5)) return;
            mark(c, ST_EXPA * 16 + 3);
            route_layer(&L, rt);
            if (c.tid == 0) mbar_arrive(c.route);
            mark(c, ST_EXPA * 16 + 0);
            if (c.cta == 0) {
                if (c.tid == 0) c.misc->distinct_total += rt->nd;
                if (p.mode == 1) {
                    for (int i = c.tid; i < c.T * m.K; i += MK_NCWARPS * 32) {
                        if (p.out_idx) p.out_idx[i] = rt->idx[i / m.K][i % m.K];
                        if (p.out_w) p.out_w[i] = rt->w[i / m.K][i % m.K];
                    }
                } else {
                    for (int i = c.tid; i < c.T * m.K; i += MK_NCWARPS * 32) {
                        if (p.trace) p.trace[(long long)l * c.T * m.K + i] = rt->idx[i / m.K][i % m.K];
                        if (p.wtrace) p.wtrace[(long long)l * c.T * m.K + i] = rt->w[i / m.K][i % m.K];
                    }
                }
            }
            ci = cons_gemv(ST_EXPA, &(L), rt, ci);
            if (!grid_sync(c, 6)) return;
        }
        // ---- routed + shared down projections (+ residual)
        mark(c, ST_EXPB * 16 + 0);
        ci = cons_gemv(ST_EXPB, &(L), rt, ci);
        if (!grid_sync(c, 7)) return;
    }
    if (p.mode == 1) {
        long long n = (long long)c.T * m.H;
        long long b = n * c.cta / c.G, e = n * (c.cta + 1) / c.G;
        for (long long i = b + c.tid; i < e; i += MK_NCWARPS * 32) p.hidden_out[i] = from_fx(__ldcg(m.res + i));
        if (c.cta == 0 && c.tid == 0) c.ctrl->epoch = c.misc->base + (unsigned long long)c.misc->nbar * c.G;
        return;
    }
    // ---- final norm + LM head
    {
        ActSrc a{m.res, nullptr, m.H, m.final_norm};
        build_frags(a, allH);
        ssq_block(c, 2);
        bar_consumers();
        ci = cons_gemv(ST_LM, &(c.misc->L[0]), &c.rt[0], ci);
        if (!grid_sync(c, 8)) return;
    }
    // ---- logits, per-CTA argmax candidates
    compute_inv_rms(c, 2);
    bar_consumers();
    {
        float *bv = reinterpret_cast<float *>(c.sm + SM_SCRATCH);
        int *bi = reinterpret_cast<int *>(c.sm + SM_SCRATCH + 4096);
        int b, e;
        split_range(m.V, c.G, c.cta, b, e);
        float best[MK_MAXT];
        int besti[MK_MAXT];
        // sampling: running maximum and sum of 2^(y - max) of y = logit * log2(e) / t
        const bool samp = p.temperature > 0.f;
        const float kt = samp ? 1.4426950408889634f / p.temperature : 0.f;
        float smx[MK_MAXT], ssum[MK_MAXT];
#pragma unroll
        for (int t = 0; t < MK_MAXT; ++t) {
            best[t] = -CUDART_INF_F;
            besti[t] = 0x7fffffff;
            smx[t] = -CUDART_INF_F;
            ssum[t] = 0.f;
        }
        for (int v0 = b + c.tid; v0 < e; v0 += 4 * MK_NCWARPS * 32) {
            long long raw[4][MK_MAXT];
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4) {
                int v = v0 + u4 * MK_NCWARPS * 32;
#pragma unroll
                for (int t = 0; t < MK_MAXT; ++t)
                    raw[u4][t] = (v < e && t < c.T) ? __ldcg(m.logit_acc + (long long)t * m.V + v) : 0;
            }
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4) {
                int v = v0 + u4 * MK_NCWARPS * 32;
                if (v >= e) break;
#pragma unroll
                for (int t = 0; t < MK_MAXT; ++t) {
                    if (t >= c.T) break;
                    float lg = from_fx(raw[u4][t]) * c.misc->inv_rms[2][t];
                    __stcs(p.out_logits + (long long)t * m.V + v, lg);
                    if (lg > best[t] || (lg == best[t] && v < besti[t])) {
                        best[t] = lg;
                        besti[t] = v;
                    }
                    if (samp) {
                        const float y = lg * kt;
                        if (y > smx[t]) {
                            ssum[t] = ssum[t] * exp2f(smx[t] - y) + 1.f;
                            smx[t] = y;
                        } else {
                            ssum[t] += exp2f(y - smx[t]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < MK_MAXT; ++t) {
            float bb = best[t];
            int bi2 = besti[t];
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                float ob = __shfl_xor_sync(0xffffffffu, bb, o);
                int oi = __shfl_xor_sync(0xffffffffu, bi2, o);
                if (ob > bb || (ob == bb && oi < bi2)) {
                    bb = ob;
                    bi2 = oi;
                }
            }
            if (c.lane == 0 && t < c.T) {
                bv[t * 8 + c.warp] = bb;
                bi[t * 8 + c.warp] = bi2;
            }
        }
        float *sv = reinterpret_cast<float *>(c.sm + SM_SCRATCH + 12288);  // [T][8] max, [T][8] sum
        if (samp) {
#pragma unroll
            for (int t = 0; t < MK_MAXT; ++t) {
                float mx = smx[t], sm = ssum[t];
#pragma unroll
                for (int o = 16; o; o >>= 1) lse_fold(mx, sm, __shfl_xor_sync(0xffffffffu, mx, o),
                                                      __shfl_xor_sync(0xffffffffu, sm, o));
                if (c.lane == 0 && t < c.T) {
                    sv[t * 8 + c.warp] = mx;
                    sv[64 + t * 8 + c.warp] = sm;
                }
            }
        }
        bar_consumers();
        if (c.tid < c.T) {
            int t = c.tid;
            float best = -CUDART_INF_F;
            int besti = 0x7fffffff;
            for (int w = 0; w < MK_NCWARPS; ++w) {
                float ob = bv[t * 8 + w];
                int oi = bi[t * 8 + w];
                if (ob > best || (ob == best && oi < besti)) {
                    best = ob;
                    besti = oi;
                }
            }
            __stcg(m.cand_v + c.cta * MK_MAXT + t, best);
            __stcg(m.cand_i + c.cta * MK_MAXT + t, besti);
            if (samp) {
                float mx = -CUDART_INF_F, sm = 0.f;
                for (int w = 0; w < MK_NCWARPS; ++w) lse_fold(mx, sm, sv[t * 8 + w], sv[64 + t * 8 + w]);
                __stcg(m.cand_m + c.cta * MK_MAXT + t, mx);
                __stcg(m.cand_s + c.cta * MK_MAXT + t, sm);
            }
        }
    }
    if (!grid_sync(c, 9)) return;
    int n_samp = -1;
    if (p.temperature > 0.f) n_samp = sample_verify_step();
    if (c.cta == 0) {
        int *am = reinterpret_cast<int *>(c.sm + SM_SCRATCH + 8192);
        if (c.tid < c.T) {
            int t = c.tid;
            float best = -CUDART_INF_F;
            int besti = 0x7fffffff;
            for (int k = 0; k < c.G; ++k) {
                float ob = __ldcg(m.cand_v + k * MK_MAXT + t);
                int oi = __ldcg(m.cand_i + k * MK_MAXT + t);
                if (ob > best || (ob == best && oi < besti)) {
                    best = ob;
                    besti = oi;
                }
            }
            am[t] = besti;
            if (p.out_argmax) p.out_argmax[t] = besti;
        }
        bar_consumers();
        if (c.tid == 0) {
            int n = 0;
            for (int i = 1; i < c.T; ++i) {
                if (__ldg(p.tokens + i) == am[i - 1]) n = i;
                else break;
            }
            if (n_samp >= 0) n = n_samp;
            *p.out_accepted = n;
            Ctrl *k = c.ctrl;
            k->steps += 1;
            k->accepted_sum += n;
            k->distinct_sum += c.misc->distinct_total;
            k->last_accepted = n;
            k->last_distinct = c.misc->distinct_total;
            k->epoch = c.misc->base + (unsigned long long)c.misc->nbar * c.G;
        }
    }
}

__global__ void __launch_bounds__(MK_THREADS, 1) mk_step_kernel(const __grid_constant__ Params p) {
    unsigned char *smem = smem_base();
    MiscSm *misc = reinterpret_cast<MiscSm *>(smem + SM_MISC);
    const DModel *gm = p.m;
    // launch parameters, model block and first layer's descriptors into shared memory
    {
        const int np = (int)(sizeof(Params) / 4);
        for (int i = threadIdx.x; i < np; i += blockDim.x)
            reinterpret_cast<uint32_t *>(&misc->pc)[i] = reinterpret_cast<const uint32_t *>(&p)[i];
        const int nw = (int)(sizeof(DModel) / 4);
        for (int i = threadIdx.x; i < nw; i += blockDim.x)
            reinterpret_cast<uint32_t *>(&misc->m)[i] = __ldg(reinterpret_cast<const uint32_t *>(gm) + i);
        const int nl = (int)(sizeof(DLayer) / 4);
        const DLayer *l0 = gm->layers + (p.mode ? p.layer : 0);
        for (int i = threadIdx.x; i < nl; i += blockDim.x)
            reinterpret_cast<uint32_t *>(&misc->L[0])[i] = __ldg(reinterpret_cast<const uint32_t *>(l0) + i);
    }
    if (threadIdx.x == 0) {
        uint64_t *full = reinterpret_cast<uint64_t *>(smem + SM_BAR), *empty = full + MK_RING,
                 *route = empty + MK_RING;
        for (int i = 0; i < MK_RING; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], MK_NCWARPS);
        }
        mbar_init(route, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        misc->abort = 0;
        misc->distinct_total = 0;
        misc->nbar = 0;
        misc->nmark = 0;
        misc->par = 0;
        misc->p = &misc->pc;
        Ctrl *ctrl = gm->ctrl;
        // validate the step's inputs (every CTA reaches the same verdict)
        const int P = gm->P;
        int ctx = __ldg(p.positions);
        int ok = (*(volatile int *)&ctrl->abort == 0) ? 1 : 0;
        for (int t = 0; t < p.T; ++t)
            if (__ldg(p.positions + t) != ctx + t) ok = 0;
        // entry points that stage per-position tables on the host (the RoPE rows
        // of the allocation-free layer call) pass the ctx they staged for
        if (p.host_ctx1 != 0 && ctx != p.host_ctx1 - 1) ok = 0;
        if (ctx < 0 || (long long)ctx + p.T > (long long)gm->max_pages * P) ok = 0;
        if (ok) {
            int np = (ctx + p.T + P - 1) / P;
            for (int j = 0; j < np; ++j) {
                int ph = __ldg(p.page_table + j);
                if (ph < 0 || ph >= p.n_pages) ok = 0;
            }
        }
        if (ok && p.mode == 0) {
            for (int t = 0; t < p.T; ++t) {
                int tk = __ldg(p.tokens + t);
                if (tk < 0 || tk >= gm->V) ok = 0;
            }
        }
        misc->valid = ok;
        misc->ctx = ok ? ctx : 0;
        const int ncp = (misc->ctx + P - 1) / P;
        misc->nsplit = min(min((int)gridDim.x / gm->Hkv, (ncp + 1 + MK_ATT_MIN_PAGES - 1) / MK_ATT_MIN_PAGES),
                           MK_MAXSPLIT);
        misc->base = *(volatile unsigned long long *)&ctrl->epoch;
    }
    __syncthreads();
    if (!misc->valid) {
        Ctrl *ctrl = gm->ctrl;
        if (blockIdx.x == 0 && threadIdx.x == 0 && *(volatile int *)&ctrl->abort == 0) {
            atomicCAS(&ctrl->status, 0, (int)MK_ERR_BAD_INPUT);
            atomicExch(&ctrl->abort, 1);
        }
        return;
    }
    {
        // the launch's split of the non-routed stages, one stage per warp
        const int st = threadIdx.x >> 5;
        if ((threadIdx.x & 31) == 0 && (st == ST_QKV || st == ST_O || st == ST_ROUTER || st == ST_SHA ||
                                        (st == ST_LM && p.mode == 0)))
            stage_seed(misc->seed[st], make_ctx(), st, misc->L[0], 0);
        if (threadIdx.x == 32) launch_masks();
        __syncthreads();
    }
    if ((threadIdx.x >> 5) == MK_NCWARPS) {
        if ((threadIdx.x & 31) < MK_PLANES) producer();
        __syncwarp();
    } else {
        consumer();
    }
}

}  // namespace

#if MK_F32_MODEL
#define MK_SFX(x) x##_f32
#else
#define MK_SFX(x) x##_lp
#endif

cudaError_t MK_SFX(mk_kernel_setup)(size_t smem) {
    return cudaFuncSetAttribute(mk_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t MK_SFX(mk_launch)(const Params &p, int grid, size_t smem, cudaStream_t s) {
    void *args[] = {(void *)&p};
    return cudaLaunchCooperativeKernel((const void *)mk_step_kernel, dim3(grid), dim3(MK_THREADS), args, smem, s);
}

int MK_SFX(mk_kernel_max_blocks)(size_t smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, mk_step_kernel, MK_THREADS, smem) != cudaSuccess) return -1;
    return n;
}
