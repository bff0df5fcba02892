// Sampling verification with point-mass drafts (HyperQwen context-lookup
// article, closing paragraph of "lookup 草稿的原理：三步走": for a sampled
// request each drafted position is a point mass on its proposed token, which
// the standard speculative rejection sampler accepts as a proposal, so the
// outputs follow plain sampling from the target).
//
// Per request b and row r < L_b the target is p_r = softmax(x_r * t_b), with
// t_b the request's inverse temperature.  The draft c = blk[r + 1] is
// accepted iff u_acc[b][r] < p_r(c); the first rejected row emits an
// inverse-CDF sample of p_r without c (the residual max(p_r - point mass, 0),
// normalised) drawn with u_smp[b][r]; a block whose L_b - 1 drafts are all
// accepted emits a sample of p_{L_b - 1}.  A draft outside [0, V) (the
// sentinel) is rejected and its row's whole p is sampled.
//
// The work is HBM-bound: every verified row is read once.  Each row is cut
// into segments of kSegElems elements; the grid takes an even share of the
// flat list of (request, row, segment) triples.  Each thread keeps, in base
// 2, a running maximum m of z = x * t * log2(e) and the sum s = sum 2^(z - m)
// over its strided vectors of a segment (one fused multiply-add and one
// hardware exp2 per element: the PTX ex2.approx.ftz.f32 instruction, whose
// relative error the PTX ISA bounds by 2^-22); each warp combines its 32
// threads' pairs with shuffles in a fixed order and stores one (m, s) pair
// per segment and warp in the scratch, so no barrier is needed per segment.  When a CTA leaves a request it adds the
// number of that request's segments it finished to the request's counter;
// the CTA that completes the count finishes the request: it combines the
// pairs of each row in a fixed order, decides all acceptances at once, finds
// the segment that holds the sample from the pairs and the token inside it by
// reading that one segment again.  Every reduction has a fixed order, so the
// results do not depend on the grid or on timing.  k_sample serves the
// stateless entry point; k_sample_step, fused with the token commit, starts
// streaming predicted rows before the proposal launch it depends on ends.
// k_sample_fx and k_sample_step_fx are the same two on weights defined as
// integers (clk_verify_sample_exact*, the section "Exact sampling" below),
// whose decisions another implementation of the definition reproduces bit
// for bit.
#include <algorithm>
#include <atomic>

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "clk.h"
#include "clk_device.cuh"
#include "clk_host.h"

namespace clk {
namespace {

#ifndef CLK_SAMPLE_CTAS
#define CLK_SAMPLE_CTAS 4  // resident CTAs per SM the kernel is compiled for
#endif
constexpr int kSThreads = 256;
constexpr int kSWarpsPerCta = kSThreads / 32;
constexpr int kSUnroll = 4;
#ifndef CLK_SAMPLE_SEG
#define CLK_SAMPLE_SEG 16384
#endif
constexpr int64_t kSegElems = CLK_SAMPLE_SEG;  // elements per segment
static_assert(kSegElems % (8 * kSUnroll * kSThreads) == 0, "a segment is whole groups of vectors");

struct SampleArgs {
    const void* logits;
    int64_t row_stride;  // elements
    int64_t req_stride;  // elements
    int32_t V;
    int32_t B;
    int32_t S;            // segments per row
    const int32_t* block;
    const int32_t* len;
    const int32_t* len_hint;  // fused: predicted block lengths (may be null)
    const float* inv_temp;  // [B]
    const float* uniform;   // [B][16][2]
    int32_t* accept;
    int32_t* emitted;
    int32_t* out_tok;
    uint32_t* done;  // [B] segments finished per request
    float2* part;    // [B][16][S][kSWarpsPerCta] (m, s) per warp
    const int32_t* slots;  // fused with the commit only: the requests' slots
    int32_t late;          // fused: trailing CTAs that start behind the proposal launch (0: none)
    int32_t paired;        // fused: scratch in two halves; the next launch is let go after the wait
};

__device__ __forceinline__ bool len_valid(int32_t l) { return l >= 1 && l <= kBlock; }
__device__ __forceinline__ bool temp_valid(float t) { return t > 0.0f && t < INFINITY; }

// Rows a request contributes: L_b for a valid length and temperature, else 0.
__device__ __forceinline__ int32_t sample_rows(const SampleArgs& a, int32_t b)
{
    const int32_t l = a.len[b];
    return (len_valid(l) && temp_valid(a.inv_temp[b])) ? l : 0;
}

template <int DT>
struct SElem;
template <>
struct SElem<CLK_DTYPE_BF16> {
    using T = uint16_t;
    static constexpr int W = 8;  // elements per 16-byte vector
    __device__ static float value(T x) { return __uint_as_float((uint32_t)x << 16); }
    // maximum of the 8 values by packed bf16x2 maxima
    __device__ static float vmax(const uint4& v)
    {
        const __nv_bfloat162 m = __hmax2(__hmax2(as2(v.x), as2(v.y)), __hmax2(as2(v.z), as2(v.w)));
        return fmaxf(__low2float(m), __high2float(m));
    }
    __device__ static __nv_bfloat162 as2(uint32_t w)
    {
        __nv_bfloat162 r;
        memcpy(&r, &w, 4);
        return r;
    }
    __device__ static void unpack(const uint4& v, float* f)
    {
        f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xFFFF0000u);
        f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xFFFF0000u);
        f[4] = __uint_as_float(v.z << 16); f[5] = __uint_as_float(v.z & 0xFFFF0000u);
        f[6] = __uint_as_float(v.w << 16); f[7] = __uint_as_float(v.w & 0xFFFF0000u);
    }
};
template <>
struct SElem<CLK_DTYPE_F32> {
    using T = float;
    static constexpr int W = 4;
    __device__ static float value(T x) { return x; }
    __device__ static float vmax(const uint4& v)
    {
        return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)), fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
    __device__ static void unpack(const uint4& v, float* f)
    {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
};

// 2^x by the hardware's base-2 exponential (flushes results below 2^-126
// to zero: weights that small against the maximum do not count).
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kLog2e = 1.4426950408889634f;

// Running (max, sum of 2^(z - max)) of a set of values z (base 2).
struct MS {
    float m;
    float s;
};

__device__ __forceinline__ MS ms_empty() { return MS{-INFINITY, 0.0f}; }

// The pair of the union of two sets.
__device__ __forceinline__ MS ms_merge(MS a, MS b)
{
    if (b.s == 0.0f) return a;
    if (a.s == 0.0f) return b;
    const float m = fmaxf(a.m, b.m);
    return MS{m, a.s * ex2(a.m - m) + b.s * ex2(b.m - m)};
}

// Two floats in one 64-bit register pair, for the packed f32x2 arithmetic
// (fma.rn.f32x2, add.rn.f32x2: two independent float operations each,
// rounded as the scalar ones).
__device__ __forceinline__ unsigned long long pk(float lo, float hi)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void pk_split(unsigned long long v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long x, unsigned long long y, unsigned long long z)
{
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(x), "l"(y), "l"(z));
    return r;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long x, unsigned long long y)
{
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(y));
    return r;
}

// Sum of the W weights 2^(x_i c - m) of one vector, in pairs, then the two
// halves.
template <int DT>
__device__ __forceinline__ float vec_weights(const float* f, float c, float m)
{
    const unsigned long long c2 = pk(c, c), nm2 = pk(-m, -m);
    unsigned long long acc = 0ull;  // (+0, +0)
#pragma unroll
    for (int i = 0; i < SElem<DT>::W; i += 2) {
        float z0, z1;
        pk_split(fma2(pk(f[i], f[i + 1]), c2, nm2), z0, z1);
        acc = add2(acc, pk(ex2(z0), ex2(z1)));
    }
    float a0, a1;
    pk_split(acc, a0, a1);
    return a0 + a1;
}

// Weights above this (relative to the running maximum) trigger a rescale;
// below it the sum cannot overflow (float reaches 2^128).
constexpr float kRescaleAt = 18446744073709551616.0f;  // 2^64

// Adds the W values z_i = x_i * c of one vector (c = t log2 e > 0).  The
// running maximum is raised lazily: the weights are taken against the
// current m, and only a vector whose weights sum past 2^64 (or to inf or
// NaN: the first vector, where m is still -inf) raises m to its own maximum
// and is weighed again.  The pair still means s = sum 2^(z - m) exactly as
// before; m need not be the largest z, only within 64 of it.
template <int DT>
__device__ __forceinline__ void ms_add_vec(MS& r, const uint4& v, float c)
{
    using E = SElem<DT>;
    float f[E::W];
    E::unpack(v, f);
    float acc = vec_weights<DT>(f, c, r.m);
    if (!(acc <= kRescaleAt)) {
        const float vm = E::vmax(v) * c;
        if (vm > r.m) {
            r.s = r.s == 0.0f ? 0.0f : r.s * ex2(r.m - vm);
            r.m = vm;
        }
        if (r.m == -INFINITY) return;  // every value so far is -inf: weight 0
        acc = vec_weights<DT>(f, c, r.m);
    }
    r.s += acc;
}

// Warp-wide merge: the largest m of the lanes, each lane's sum taken
// against it, and the sums added in a fixed (butterfly) order.  Both
// partners of every exchange add the same two numbers, so every lane gets
// the same result.  A lane with s = 0 (no weight yet) adds nothing; its m is
// -inf, so it does not raise the maximum either.
__device__ __forceinline__ MS ms_warp(MS r)
{
    float m = r.m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    float s = r.s == 0.0f ? 0.0f : r.s * ex2(r.m - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    return MS{m, s};
}

// Adds one value z = x * c.
__device__ __forceinline__ void ms_add1(MS& r, float x, float c)
{
    const float z = x * c;
    if (z > r.m) {
        r.s = r.s == 0.0f ? 0.0f : r.s * ex2(r.m - z);
        r.m = z;
    }
    if (r.m != -INFINITY) r.s += ex2(fmaf(x, c, -r.m));
}

// P[b] = rows(b') summed over requests b' < b; P[B] = total.  Block-wide.
template <typename Rows>
__device__ __forceinline__ void rows_prefix(int32_t B, Rows rows, int32_t* P, int32_t* sm_warp)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t per = (B + kSThreads - 1) / kSThreads;
    const int32_t b0 = min(B, tid * per), b1 = min(B, b0 + per);
    // rows(b) is read once (it may load from global memory): kept in P[b]
    // (this thread's own entries) until the prefix overwrites it
    int32_t local = 0;
    for (int32_t b = b0; b < b1; ++b) {
        const int32_t r = rows(b);
        P[b] = r;
        local += r;
    }
    int32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sm_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int32_t s = lane < kSWarpsPerCta ? sm_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < kSWarpsPerCta) sm_warp[lane] = s;
    }
    __syncthreads();
    int32_t run = (incl - local) + (warp > 0 ? sm_warp[warp - 1] : 0);
    for (int32_t b = b0; b < b1; ++b) {
        const int32_t r = P[b];
        P[b] = run;
        run += r;
    }
    if (tid == kSThreads - 1) P[B] = sm_warp[kSWarpsPerCta - 1];
    __syncthreads();
}

// P[b] = rows of requests b' < b; P[B] = total.  Block-wide.
__device__ __forceinline__ void sample_prefix(const SampleArgs& a, int32_t* P, int32_t* sm_warp)
{
    rows_prefix(a.B, [&a](int32_t b) { return sample_rows(a, b); }, P, sm_warp);
}

// Largest b with P[b] <= ri.
__device__ __forceinline__ int32_t sample_owner(const int32_t* P, int32_t B, int64_t ri)
{
    int32_t b = 0, top = B;
    while (b < top) {
        const int32_t mid = (b + top + 1) >> 1;
        if (P[mid] <= ri) b = mid; else top = mid - 1;
    }
    return b;
}

__device__ __forceinline__ float2* part_of(const SampleArgs& a, int32_t b, int32_t r, int32_t seg)
{
    return a.part + (((int64_t)b * kBlock + r) * a.S + seg) * kSWarpsPerCta;
}

// Segment k (flat) of request b: the row's first byte and the segment's
// range in units (vectors on the vector path, elements otherwise).
template <int DT, bool VEC>
__device__ __forceinline__ void seg_range(const SampleArgs& a, const int32_t* P, int32_t b, int32_t roff, int64_t k,
                                          const char*& row, int32_t& u0, int32_t& u1, int32_t& r, int32_t& sg)
{
    using E = SElem<DT>;
    constexpr int W = VEC ? E::W : 1;
    const int64_t ri = k / a.S;
    sg = (int32_t)(k - ri * a.S);
    r = roff + (int32_t)(ri - P[b]);
    row = static_cast<const char*>(a.logits) +
          ((int64_t)b * a.req_stride + (int64_t)r * a.row_stride) * (int64_t)sizeof(typename E::T);
    const int64_t e0 = (int64_t)sg * kSegElems, e1 = min(e0 + kSegElems, (int64_t)a.V);
    u0 = (int32_t)(e0 / W);
    u1 = (int32_t)(e1 / W);
}

// Streams segments [k0, k1) of request b (flat segment k is segment k % S of
// the request's row roff + k / S - P[b]) and stores one (m, s) pair per
// segment and warp.  Vector path: two groups of kSUnroll 16-byte loads per
// thread alternate, and the next segment's first group is issued before the
// current segment's last group is reduced.  The segment and row advance
// incrementally (segments of a request are consecutive: row-major).
template <int DT>
__device__ __forceinline__ void stream_vec(const SampleArgs& a, const int32_t* P, int32_t b, int32_t roff, int64_t k0,
                                           int64_t k1)
{
    using E = SElem<DT>;
    constexpr int32_t SV = (int32_t)(kSegElems / E::W);  // vectors per full segment
    constexpr int32_t G = kSUnroll * kSThreads;          // vectors per group
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float c = a.inv_temp[b] * kLog2e;
    const int32_t vpr = a.V / E::W;
    const int64_t rsv = a.row_stride / E::W;  // row stride in vectors
    const uint4* req = reinterpret_cast<const uint4*>(static_cast<const char*>(a.logits) +
                                                     (int64_t)b * a.req_stride * (int64_t)sizeof(typename E::T));
    const int64_t ri0 = k0 / a.S;
    int32_t r = roff + (int32_t)(ri0 - P[b]);
    int32_t sg = (int32_t)(k0 - ri0 * a.S);
    int32_t left = (int32_t)(k1 - k0);  // segments still to finish, the current one included
    // current group: row `row`, vectors [g, g + G) of segment sg (which ends at e)
    const uint4* row = req + (int64_t)r * rsv;
    int32_t g = sg * SV;
    int32_t e = min(g + SV, vpr);
    MS run = ms_empty();
    uint4 X[kSUnroll], Y[kSUnroll];
#define CLK_LOAD_GROUP(D, RW, G0, E0)                                                  \
    if ((G0) + G <= (E0)) {                                                            \
        _Pragma("unroll") for (int u = 0; u < kSUnroll; ++u) D[u] = __ldcs((RW) + (G0) + tid + u * kSThreads); \
    } else {                                                                           \
        _Pragma("unroll") for (int u = 0; u < kSUnroll; ++u) {                         \
            const int32_t vi = (G0) + tid + u * kSThreads;                             \
            if (vi < (E0)) D[u] = __ldcs((RW) + vi);                                   \
        }                                                                              \
    }
#define CLK_REDUCE_GROUP(D, G0, E0)                                                    \
    if ((G0) + G <= (E0)) {                                                            \
        _Pragma("unroll") for (int u = 0; u < kSUnroll; ++u) ms_add_vec<DT>(run, D[u], c); \
    } else {                                                                           \
        _Pragma("unroll") for (int u = 0; u < kSUnroll; ++u)                           \
            if ((G0) + tid + u * kSThreads < (E0)) ms_add_vec<DT>(run, D[u], c);       \
    }
    CLK_LOAD_GROUP(X, row, g, e)
    for (int half = 0;; half ^= 1) {
        // the next group: later in this segment, or the first of the next
        const uint4* nrow = row;
        int32_t ng = g + G, ne = e, nr = r, nsg = sg;
        const bool seg_end = ng >= e;
        const bool more = !seg_end || left > 1;
        if (seg_end && more) {
            nsg = sg + 1;
            if (nsg == a.S) {
                nsg = 0;
                nr = r + 1;
                nrow = req + (int64_t)nr * rsv;
            }
            ng = nsg * SV;
            ne = min(ng + SV, vpr);
        }
        if (half == 0) {
            if (more) { CLK_LOAD_GROUP(Y, nrow, ng, ne) }
            CLK_REDUCE_GROUP(X, g, e)
        } else {
            if (more) { CLK_LOAD_GROUP(X, nrow, ng, ne) }
            CLK_REDUCE_GROUP(Y, g, e)
        }
        if (seg_end) {
            const MS w = ms_warp(run);
            if (lane == 0) part_of(a, b, r, sg)[warp] = make_float2(w.m, w.s);
            run = ms_empty();
            --left;
        }
        if (!more) break;
        row = nrow;
        g = ng;
        e = ne;
        r = nr;
        sg = nsg;
    }
#undef CLK_LOAD_GROUP
#undef CLK_REDUCE_GROUP
}

// Scalar path (rows not 16-byte aligned): one segment at a time.
template <int DT>
__device__ __forceinline__ void stream_scalar(const SampleArgs& a, const int32_t* P, int32_t b, int32_t roff,
                                              int64_t k0, int64_t k1)
{
    using E = SElem<DT>;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float c = a.inv_temp[b] * kLog2e;
    for (int64_t k = k0; k < k1; ++k) {
        const char* rowp;
        int32_t u0, u1, r, sg;
        seg_range<DT, false>(a, P, b, roff, k, rowp, u0, u1, r, sg);
        const typename E::T* row = reinterpret_cast<const typename E::T*>(rowp);
        MS run = ms_empty();
        for (int32_t i = u0 + tid; i < u1; i += kSThreads) ms_add1(run, E::value(row[i]), c);
        const MS w = ms_warp(run);
        if (lane == 0) part_of(a, b, r, sg)[warp] = make_float2(w.m, w.s);
    }
}

struct FinSmem {
    float m[kBlock], s[kBlock];  // each row's combined pair
    float xc[kBlock];            // each row's draft logit
    float ex;                    // weight of the removed draft
    unsigned long long tgt;      // the draw's target inside the chosen segment (fixed point)
    int32_t a, excl, seg, tok, cross;
    unsigned long long wsum[kSWarpsPerCta];
    int32_t lastw[kSWarpsPerCta];  // each warp's last element of positive weight
    int32_t out[kBlock];  // the emitted tokens (fused: committed)
    int32_t flag[3];
};

// Request b is complete (all of its segments' pairs are stored): decide the
// drafts, draw the token, write the outputs, rewind the counter.  Block-wide.
template <int DT, bool FUSED>
__device__ __noinline__ void sample_finish(const SampleArgs& a, const LookupDev& Ldev, int32_t b, FinSmem& fs)
{
    using E = SElem<DT>;
    const unsigned full = 0xFFFFFFFFu;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t L = a.len[b], S = a.S, V = a.V;
    const float cz = a.inv_temp[b] * kLog2e;  // z = x * cz, weights 2^(z - m)
    const typename E::T* base = static_cast<const typename E::T*>(a.logits) + (int64_t)b * a.req_stride;
    __threadfence();
    // Each row's pair: 16 threads per row (row = tid / 16), each merging the
    // row's segment pairs sub, sub + 16, ... in order, then a butterfly over
    // the 16.  Warp 0 also loads every draft's logit in the same round trip.
    {
        const int32_t r = tid >> 4, sub = tid & 15;
        float xc = 0.0f;
        if (warp == 0 && lane < L - 1) {
            const int32_t c = a.block[(int64_t)b * kBlock + lane + 1];
            if (c >= 0 && c < V) xc = E::value(base[(int64_t)lane * a.row_stride + c]);
        }
        MS acc = ms_empty();
        if (r < L) {
            const float2* pp = part_of(a, b, r, 0);
            const int32_t n = S * kSWarpsPerCta;
#pragma unroll 8
            for (int32_t i = sub; i < n; i += 16) {
                const float2 q = __ldcg(pp + i);
                acc = ms_merge(acc, MS{q.x, q.y});
            }
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
            MS q;
            q.m = __shfl_xor_sync(full, acc.m, o);
            q.s = __shfl_xor_sync(full, acc.s, o);
            acc = (sub & o) ? ms_merge(q, acc) : ms_merge(acc, q);
        }
        if (sub == 0 && r < L) {
            fs.m[r] = acc.m;
            fs.s[r] = acc.s;
        }
        if (warp == 0 && lane < kBlock) fs.xc[lane] = xc;
    }
    __syncthreads();
    // Acceptance of every draft at once (lane r: row r's draft blk[r + 1]).
    if (warp == 0) {
        const bool has = lane < L - 1;
        const int32_t c = has ? a.block[(int64_t)b * kBlock + lane + 1] : CLK_SENT;
        const bool inv = c >= 0 && c < V;
        float ec = 0.0f;
        if (has && inv) ec = ex2(fmaf(fs.xc[lane], cz, -fs.m[lane]));
        const float p = has ? ec / fs.s[lane] : 0.0f;
        const float ua = has ? a.uniform[((int64_t)b * kBlock + lane) * 2] : 1.0f;
        const unsigned rej = __ballot_sync(full, has && !(ua < p));
        const int32_t acc_n = rej ? __ffs(rej) - 1 : L - 1;
        if (lane == acc_n) {
            fs.a = acc_n;
            fs.excl = (has && inv) ? c : -1;
            fs.ex = (has && inv) ? ec : 0.0f;
        }
    }
    __syncthreads();
    const int32_t ra = fs.a, excl = fs.excl;
    const float mra = fs.m[ra];
    // The segment holding the draw.  The draw's prefix arithmetic is exact:
    // sums of more than a few weights are scaled to 64-bit fixed point (2^61
    // for the row's sum) and added as integers, so the long running sums
    // round nowhere; token widths in a large vocabulary are far below
    // float32's resolution of a sum of the whole row.  Segment weights (from the stored pairs,
    // relative to the row's maximum, the removed draft taken out of its
    // segment) are summed once for the total and again, in order, to find
    // the segment whose running sum passes u * total.
    const float sc = 2305843009213693952.0f / fmaxf(fs.s[ra], 1.0f);  // 2^61 / row sum
    if (warp == 0) {
        const float2* pp = part_of(a, b, ra, 0);
        const int32_t exseg = excl >= 0 ? (int32_t)(excl / kSegElems) : -1;
        const unsigned long long qex = __float2ull_rn(fs.ex * sc);
        auto seg_weight = [&](int32_t k) -> unsigned long long {
            if (k >= S) return 0ull;
            float w = 0.0f;
            for (int i = 0; i < kSWarpsPerCta; ++i) {
                const float2 q = __ldcg(pp + (int64_t)k * kSWarpsPerCta + i);
                if (q.y > 0.0f) w += q.y * ex2(q.x - mra);
            }
            unsigned long long qw = __float2ull_rn(w * sc);
            if (k == exseg) qw = qw > qex ? qw - qex : 0ull;
            return qw;
        };
        unsigned long long total = 0ull;
        for (int32_t k0 = 0; k0 < S; k0 += 32) {
            unsigned long long w = seg_weight(k0 + lane);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(full, w, o);
            total += w;
        }
        const unsigned long long target =
            __double2ull_rd((double)a.uniform[((int64_t)b * kBlock + ra) * 2 + 1] * (double)total);
        unsigned long long carry = 0ull, before = 0ull;
        int32_t found = -1, lastpos = -1;
        for (int32_t k0 = 0; k0 < S && found < 0; k0 += 32) {
            const int32_t k = k0 + lane;
            const unsigned long long w = seg_weight(k);
            unsigned long long incl = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(full, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned cross = __ballot_sync(full, k < S && carry + incl > target);
            const unsigned pos = __ballot_sync(full, k < S && w > 0ull);
            if (pos) lastpos = k0 + 31 - __clz(pos);
            if (cross) {
                const int32_t l = __ffs(cross) - 1;
                found = k0 + l;
                before = carry + __shfl_sync(full, incl - w, l);
            }
            carry += __shfl_sync(full, incl, 31);
        }
        if (lane == 0) {
            fs.seg = found >= 0 ? found : lastpos;
            fs.tgt = found >= 0 ? target - before : ~0ull;  // no crossing: the last positive weight
        }
    }
    __syncthreads();
    // Inside the segment, in chunks of kChunk elements: each thread weighs a
    // contiguous run of kRun elements (its loads issued together), a
    // block-wide exclusive scan of the runs' sums places the target, and the
    // thread whose run crosses it walks its weights.
    constexpr int32_t kRun = 16;
    constexpr int32_t kChunk = kRun * kSThreads;
    const int32_t sg = fs.seg;
    const typename E::T* row = base + (int64_t)ra * a.row_stride;
    const int64_t s0 = sg < 0 ? 0 : (int64_t)sg * kSegElems;
    const int64_t s1 = sg < 0 ? 0 : min(s0 + kSegElems, (int64_t)V);
    unsigned long long tgt = fs.tgt;
    int64_t lastv = -1;  // this thread's last element of positive weight
    if (tid == 0) fs.tok = CLK_SENT;
    for (int64_t c0 = s0; c0 < s1; c0 += kChunk) {
        const int64_t v0 = c0 + (int64_t)tid * kRun;
        float wv[kRun];
        float ownf = 0.0f;  // 16 weights: float is exact enough for one run
#pragma unroll
        for (int i = 0; i < kRun; ++i) {
            const int64_t v = v0 + i;
            const bool in = v < s1 && v != excl;
            const float x = v < s1 ? E::value(row[v]) : 0.0f;
            wv[i] = in ? ex2(fmaf(x, cz, -mra)) : 0.0f;
            ownf += wv[i];
            if (wv[i] > 0.0f) lastv = v;
        }
        const unsigned long long own = __float2ull_rn(ownf * sc);
        unsigned long long incl = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(full, incl, o);
            if (lane >= o) incl += y;
        }
        __syncthreads();  // the previous chunk's sums have been read
        if (lane == 31) fs.wsum[warp] = incl;
        if (tid == 0) fs.cross = -1;
        __syncthreads();
        unsigned long long pre = incl - own, tot = 0ull;
        for (int w = 0; w < kSWarpsPerCta; ++w) {
            if (w < warp) pre += fs.wsum[w];
            tot += fs.wsum[w];
        }
        if (tgt < tot) {  // the same decision in every thread
            // the crossing run: the last one of positive weight that starts
            // at or before the target (one exists: the first positive run
            // starts at 0 <= target)
            if (own > 0ull && pre <= tgt) atomicMax(&fs.cross, tid);
            __syncthreads();
            if (tid == fs.cross) {
                unsigned long long run = pre;
                int64_t tok = lastv;
#pragma unroll
                for (int i = 0; i < kRun; ++i) {
                    run += __float2ull_rn(wv[i] * sc);
                    if (wv[i] > 0.0f && run > tgt) {
                        tok = v0 + i;
                        break;
                    }
                }
                fs.tok = (int32_t)tok;
            }
            break;
        }
        tgt -= tot;
    }
    __syncthreads();
    if (fs.tok == CLK_SENT) {
        // no crossing (rounding, or the target past the segment): the
        // segment's last element of positive weight
        const unsigned has = __ballot_sync(full, lastv >= 0);
        __syncthreads();
        if (has && lane == 31 - __clz(has)) fs.lastw[warp] = (int32_t)lastv;
        else if (lane == 0 && !has) fs.lastw[warp] = -1;
        __syncthreads();
        if (tid == 0) {
            for (int w = kSWarpsPerCta - 1; w >= 0; --w) {
                const int32_t v = fs.lastw[w];
                if (v >= 0) {
                    fs.tok = v;
                    break;
                }
            }
        }
        __syncthreads();
    }
    if (tid < kBlock) {
        const int32_t r = tid;
        const int32_t out = r < fs.a ? a.block[(int64_t)b * kBlock + r + 1] : (r == fs.a ? fs.tok : CLK_SENT);
        a.out_tok[(int64_t)b * kBlock + r] = out;
        fs.out[r] = out;
    }
    if (tid == 0) {
        a.accept[b] = fs.a;
        a.emitted[b] = fs.a + 1;
        a.done[b] = 0u;
    }
    __syncthreads();
    if (FUSED) {
        const int32_t slot = a.slots[b];
        if (slot < 0 || slot >= Ldev.max_slots) {
            if (tid == 0) latch(Ldev.status, CLK_EINVAL, b);
        } else {
            block_commit_tokens(Ldev, slot, fs.out, fs.a + 1, fs.flag);
        }
        __syncthreads();
    }
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kSThreads, CLK_SAMPLE_CTAS) k_sample(SampleArgs a, LookupDev Ldev)
{
    extern __shared__ int32_t P[];  // B + 1
    __shared__ int32_t sm_warp[kSWarpsPerCta];
    __shared__ int32_t sm_last;
    __shared__ FinSmem fs;
    const int tid = threadIdx.x;
    const int32_t B = a.B;
    sample_prefix(a, P, sm_warp);
    // Requests with no rows (invalid length or temperature): empty result.
    if (blockIdx.x == 0) {
        for (int32_t b = tid; b < B; b += kSThreads) {
            if (sample_rows(a, b) != 0) continue;
            for (int r = 0; r < kBlock; ++r) a.out_tok[(int64_t)b * kBlock + r] = CLK_SENT;
            a.accept[b] = 0;
            a.emitted[b] = 0;
        }
    }
    const int64_t S = a.S;
    const int64_t N = (int64_t)P[B] * S;
    const int64_t lo = N * blockIdx.x / gridDim.x;
    const int64_t hi = N * (blockIdx.x + 1) / gridDim.x;
    int64_t k = lo;
    while (k < hi) {
        const int32_t b = sample_owner(P, B, k / S);
        const int64_t k1 = min(hi, (int64_t)P[b + 1] * S);
        if (VEC) stream_vec<DT>(a, P, b, 0, k, k1);
        else stream_scalar<DT>(a, P, b, 0, k, k1);
        __syncthreads();  // every warp's pairs are stored
        if (tid == 0) {
            __threadfence();
            const uint32_t n = (uint32_t)(k1 - k);
            const uint32_t need = (uint32_t)(P[b + 1] - P[b]) * (uint32_t)S;
            sm_last = atomicAdd(a.done + b, n) + n == need;
        }
        __syncthreads();
        if (sm_last) sample_finish<DT, false>(a, Ldev, b, fs);
        k = k1;
    }
}

// ---------------------------------------------------------------------------
// Exact sampling (clk_verify_sample_exact): the same rule on weights defined
// as integers, so that every acceptance and every draw is an integer
// comparison and the result is a fixed function of the logits, uniforms and
// drafts (where floating point decides an integer, the precision is part of
// the definition: float32 with fused multiply-adds, then integers).
//
// s = fl32(t * fl32(log2 e)).  A row is cut into chunks of kFxChunk entries;
// chunk k's reference is R_k = ceil(fl32(M_k * s)), M_k its largest entry.
// Entry x of chunk k weighs q = Q(d), d = fma(x, s, -R_k): for d >= -32,
// with n = rint(d) and r = d - n, f = P(r) is the degree-6 Taylor polynomial
// of 2^(r + 1/2) (coefficients sqrt(2) (ln 2)^j / j! rounded to float,
// Horner's rule with fused multiply-adds), a float in [1, 2], and
// q = floor(64 (bits(f) - bits(0.5f)) / 2^-n + 1/2), about 2^(d + 29.5);
// below -32, q = 0.  The chunk keeps S_k = sum of its q (exact) and R_k.
// Row units are 2^-12 of a unit of the row's reference R = max_k R_k: a
// chunk quantity v is U(v, e) = v 2^(12 - e), floored, with e = R - R_k, and
// the row's total is T = sum_k U(S_k, e_k).  A draft c in chunk kc (weight
// q_c) is accepted iff floor(k(u) T / 2^24) < U(q_c, e_kc), with
// k(u) = floor(u 2^24) clamped to [0, 2^24 - 1].  The draw takes
// t = floor(k(u) T' / 2^24) of the chunk totals with c's weight removed from
// its chunk, finds the chunk whose running total passes t and, inside it,
// the entry whose running sum of q passes the remainder taken back to chunk
// units.
//
// The streaming pass: each warp takes whole chunks of its CTA's share (the
// flat (request, row, chunk) list), one load per vector of the chunk, then a
// warp maximum, the weights in packed f32x2 arithmetic and a warp sum; one
// 64-bit record per chunk, (S_k << 24) | (R_k mod 2^24).  The CTA that
// completes a request's count finishes it: rows' totals from the records,
// all drafts at once, the chunk of the draw, the entry inside it.
// ---------------------------------------------------------------------------
constexpr int32_t kFxChunk = 1024;                  // entries per chunk
constexpr int32_t kFxNoRef = -(1 << 23);             // a chunk of -inf only
constexpr unsigned long long kFxBad = ~0ull;         // a chunk that cannot be weighed
constexpr float kFxZMax = 4194304.0f;                // 2^22: largest |M_k * s|
constexpr float kFxMagic = 12582912.0f;              // 1.5 * 2^23: d + magic rounds d to an integer
constexpr int32_t kFxGuard = 12;                     // row units: 2^-12 of a unit of the row's reference
constexpr int32_t kFxVMax = 4194304;                 // longest row (4096 chunks: T stays below 2^64)
#ifndef CLK_FX_CTAS
#define CLK_FX_CTAS 4  // resident CTAs per SM the exact sampler is compiled for
#endif
constexpr int kFxCtas = CLK_FX_CTAS;

// The weight polynomial's coefficients, packed twice for f32x2 arithmetic.
struct FxPoly {
    unsigned long long c2[7];
    float c[7];
};

__device__ __forceinline__ int32_t fx_ref(unsigned long long rec)
{
    return (int32_t)((uint32_t)rec << 8) >> 8;  // the low 24 bits, sign-extended
}
__device__ __forceinline__ unsigned long long fx_sum(unsigned long long rec) { return rec >> 24; }
// U(v, e): a chunk quantity in row units, e = R - R_k >= 0.
__device__ __forceinline__ unsigned long long fx_rowunits(unsigned long long v, int32_t e)
{
    if (e <= kFxGuard) return v << (kFxGuard - e);
    return e - kFxGuard >= 64 ? 0ull : v >> (e - kFxGuard);
}
// A row-unit remainder back in chunk units.
__device__ __forceinline__ unsigned long long fx_chunkunits(unsigned long long v, int32_t e)
{
    return e >= kFxGuard ? v << (e - kFxGuard) : v >> (kFxGuard - e);
}
// floor(k v / 2^24) for k < 2^24 and v < 2^62 (exact, in 64-bit parts).
__device__ __forceinline__ unsigned long long fx_mulshift(uint32_t k, unsigned long long v)
{
    return (unsigned long long)k * (v >> 24) + (((unsigned long long)k * (v & 0xFFFFFFull)) >> 24);
}
__device__ __forceinline__ uint32_t fx_unit(float u)
{
    const float v = u * 16777216.0f;
    if (!(v > 0.0f)) return 0u;
    if (v >= 16777215.0f) return 16777215u;
    return (uint32_t)v;
}

// q from f = P(r) and t = fl32(d + magic) = magic + n: v = floor(128 (bits(f)
// - bits(0.5f)) / 2^-n), -n = bits(magic) - bits(t), then q = (v + 1) / 2
// rounded down, i.e. v - v / 2.  For d below -2^22, -inf or NaN, t is no
// longer magic + n but the shift amount, read unsigned, is 32 or more, and
// the clamped funnel shift of (0:lo) gives 0.  q <= 2^29.75 + 1, so four
// weights add up below 2^32.
__device__ __forceinline__ uint32_t fx_q_bits(float f, float t)
{
    const uint32_t lo = __float_as_uint(f) * 128u + 0x80000000u;
    const uint32_t sh = 0x4B400000u - __float_as_uint(t);
    uint32_t v;
    asm("shf.r.clamp.b32 %0, %1, %2, %3;" : "=r"(v) : "r"(lo), "r"(0u), "r"(sh));
    return v - (v >> 1);
}

// The weight of one entry against its chunk's reference R.
__device__ __forceinline__ uint32_t fx_q1(float x, float s, int32_t R, const FxPoly& P)
{
    const float d = fmaf(x, s, -(float)R);
    const float t = __fadd_rn(d, kFxMagic);
    const float nf = __fadd_rn(t, -kFxMagic);
    const float r = __fadd_rn(d, -nf);
    float f = P.c[6];
#pragma unroll
    for (int j = 5; j >= 0; --j) f = fmaf(f, r, P.c[j]);
    return fx_q_bits(f, t);
}

// The weights of two entries (packed) against -R (packed in nR2).
__device__ __forceinline__ uint32_t fx_q2(unsigned long long x2, unsigned long long s2, unsigned long long nR2,
                                          const FxPoly& P)
{
    const unsigned long long d = fma2(x2, s2, nR2);
    const unsigned long long t = add2(d, pk(kFxMagic, kFxMagic));
    const unsigned long long nf = add2(t, pk(-kFxMagic, -kFxMagic));
    const unsigned long long r = fma2(nf, pk(-1.0f, -1.0f), d);  // d - nf, one rounding
    unsigned long long f = P.c2[6];
#pragma unroll
    for (int j = 5; j >= 0; --j) f = fma2(f, r, P.c2[j]);
    float f0, f1, t0, t1;
    pk_split(f, f0, f1);
    pk_split(t, t0, t1);
    return fx_q_bits(f0, t0) + fx_q_bits(f1, t1);
}

// Order-preserving int of a float (not NaN), for the warp maximum.
__device__ __forceinline__ int32_t fx_key(float x)
{
    const int32_t i = __float_as_int(x);
    return i ^ ((i >> 31) & 0x7FFFFFFF);
}
__device__ __forceinline__ float fx_warp_max(float x)
{
    const int32_t k = __reduce_max_sync(0xFFFFFFFFu, fx_key(x));
    return __int_as_float(k ^ ((k >> 31) & 0x7FFFFFFF));
}
// Sum over the warp of lane values below 2^48, exact, in 16-bit parts.
__device__ __forceinline__ unsigned long long fx_warp_sum(unsigned long long v)
{
    const uint32_t a = __reduce_add_sync(0xFFFFFFFFu, (uint32_t)v & 0xFFFFu);
    const uint32_t b = __reduce_add_sync(0xFFFFFFFFu, (uint32_t)(v >> 16) & 0xFFFFu);
    const uint32_t c = __reduce_add_sync(0xFFFFFFFFu, (uint32_t)(v >> 32) & 0xFFFFu);
    return ((unsigned long long)c << 32) + ((unsigned long long)b << 16) + a;
}

template <int DT>
struct FxVec;
template <>
struct FxVec<CLK_DTYPE_BF16> {
    __device__ static uint4 neg_inf() { return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u); }
    // the largest of a lane's 4 vectors: packed bf16 maxima over all 16 words, then the two halves
    __device__ static float vmax(const uint4 (&X)[4])
    {
        using E = SElem<CLK_DTYPE_BF16>;
        __nv_bfloat162 m = __hmax2(__hmax2(E::as2(X[0].x), E::as2(X[0].y)), __hmax2(E::as2(X[0].z), E::as2(X[0].w)));
#pragma unroll
        for (int u = 1; u < 4; ++u)
            m = __hmax2(m, __hmax2(__hmax2(E::as2(X[u].x), E::as2(X[u].y)), __hmax2(E::as2(X[u].z), E::as2(X[u].w))));
        return fmaxf(__low2float(m), __high2float(m));
    }
    // the 8 weights of one vector, in pairs, then two sums of four
    __device__ static unsigned long long weights(const uint4& v, unsigned long long s2, unsigned long long nR2,
                                                 const FxPoly& P)
    {
        const uint32_t a = fx_q2(pk(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u)), s2, nR2, P) +
                           fx_q2(pk(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u)), s2, nR2, P);
        const uint32_t b = fx_q2(pk(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u)), s2, nR2, P) +
                           fx_q2(pk(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u)), s2, nR2, P);
        return (unsigned long long)a + b;
    }
};
template <>
struct FxVec<CLK_DTYPE_F32> {
    __device__ static uint4 neg_inf() { return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u); }
    __device__ static float vmax(const uint4 (&X)[8])
    {
        using E = SElem<CLK_DTYPE_F32>;
        float m = E::vmax(X[0]);
#pragma unroll
        for (int u = 1; u < 8; ++u) m = fmaxf(m, E::vmax(X[u]));
        return m;
    }
    __device__ static unsigned long long weights(const uint4& v, unsigned long long s2, unsigned long long nR2,
                                                 const FxPoly& P)
    {
        return fx_q2(pk(__uint_as_float(v.x), __uint_as_float(v.y)), s2, nR2, P) +
               fx_q2(pk(__uint_as_float(v.z), __uint_as_float(v.w)), s2, nR2, P);
    }
};

// The record of a chunk from its maximum (warp-uniform) and its weights.
__device__ __forceinline__ unsigned long long fx_record(unsigned long long S, int32_t R)
{
    return (S << 24) | ((uint32_t)R & 0xFFFFFFu);
}

// Streams chunks [k0, k1) of request b (flat chunk k is chunk k % NC of the
// request's row roff + k / NC - P[b]): warp w takes chunks k0 + w, k0 + w + 8,
// ...
// Every lane holds 32 entries of its chunk (vector path: vectors lane + 32 u);
// weights are added in 32 bits four at a time, then in 64 bits.
template <int DT, bool VEC>
__device__ __forceinline__ void fx_stream(const SampleArgs& a, const int32_t* P, int32_t b, int32_t roff, int64_t k0,
                                          int64_t k1, const FxPoly& poly, unsigned long long* rec)
{
    using E = SElem<DT>;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t NC = a.S;
    const float s = a.inv_temp[b] * kLog2e;
    const unsigned long long s2 = pk(s, s);
    const typename E::T* req = static_cast<const typename E::T*>(a.logits) + (int64_t)b * a.req_stride;
    unsigned long long* recb = rec + (int64_t)b * kBlock * NC;
    // this warp's first chunk (one division per call), then 8 chunks on per step
    const int64_t kw = k0 + warp;
    const int64_t ri0 = kw / NC;
    int32_t ck = (int32_t)(kw - ri0 * NC);
    int32_t r = roff + (int32_t)(ri0 - P[b]);
    for (int64_t k = kw; k < k1; k += kSWarpsPerCta) {
        const typename E::T* row = req + (int64_t)r * a.row_stride;
        const int32_t e0 = ck * kFxChunk, n = min(kFxChunk, a.V - e0);  // entries of this chunk
        unsigned long long out;
        if (VEC) {
            constexpr int NV = kFxChunk / (E::W * 32);  // vectors per lane
            const uint4* rv = reinterpret_cast<const uint4*>(row + e0);
            const int32_t nvec = n / E::W;
            uint4 X[NV];
            if (nvec == NV * 32) {  // a whole chunk (all but a row's last): no bounds to test
#pragma unroll
                for (int u = 0; u < NV; ++u) X[u] = __ldcs(rv + lane + 32 * u);
            } else {
#pragma unroll
                for (int u = 0; u < NV; ++u) {
                    const int32_t vi = lane + 32 * u;
                    X[u] = vi < nvec ? __ldcs(rv + vi) : FxVec<DT>::neg_inf();
                }
            }
            float mx = fx_warp_max(FxVec<DT>::vmax(X));
            if (mx == -INFINITY) {
                out = fx_record(0ull, kFxNoRef);
            } else {
                const float y = mx * s;
                if (!(fabsf(y) <= kFxZMax)) {
                    out = kFxBad;
                } else {
                    const float R = ceilf(y);
                    const unsigned long long nR2 = pk(-R, -R);
                    unsigned long long sum = 0ull;
#pragma unroll
                    for (int u = 0; u < NV; ++u) sum += FxVec<DT>::weights(X[u], s2, nR2, poly);
                    out = fx_record(fx_warp_sum(sum), (int32_t)R);
                }
            }
        } else {
            float x[32];
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int32_t v = lane + 32 * i;
                x[i] = v < n ? E::value(row[e0 + v]) : -INFINITY;
                mx = fmaxf(mx, x[i]);
            }
            mx = fx_warp_max(mx);
            if (mx == -INFINITY) {
                out = fx_record(0ull, kFxNoRef);
            } else {
                const float y = mx * s;
                if (!(fabsf(y) <= kFxZMax)) {
                    out = kFxBad;
                } else {
                    const int32_t R = (int32_t)ceilf(y);
                    unsigned long long sum = 0ull;
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        sum += fx_q1(x[i], s, R, poly) + fx_q1(x[i + 1], s, R, poly) + fx_q1(x[i + 2], s, R, poly) +
                               fx_q1(x[i + 3], s, R, poly);
                    out = fx_record(fx_warp_sum(sum), R);
                }
            }
        }
        if (lane == 0) recb[r * NC + ck] = out;
        ck += kSWarpsPerCta;
        while (ck >= NC) {  // warp-uniform; once at most unless a row has fewer than 8 chunks
            ck -= NC;
            ++r;
        }
    }
}

// Block-wide sum of v (every thread gets it); sm holds one value per warp.
__device__ __forceinline__ unsigned long long fx_block_sum(unsigned long long v, unsigned long long* sm)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if (lane == 0) sm[warp] = v;
    __syncthreads();
    unsigned long long s = 0ull;
#pragma unroll
    for (int w = 0; w < kSWarpsPerCta; ++w) s += sm[w];
    __syncthreads();
    return s;
}

// Block-wide inclusive scan of v in thread order; total receives the sum.
__device__ __forceinline__ unsigned long long fx_block_scan(unsigned long long v, unsigned long long* sm,
                                                            unsigned long long& total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sm[warp] = incl;
    __syncthreads();
    unsigned long long pre = 0ull, tot = 0ull;
#pragma unroll
    for (int w = 0; w < kSWarpsPerCta; ++w) {
        if (w < warp) pre += sm[w];
        tot += sm[w];
    }
    __syncthreads();
    total = tot;
    return pre + incl;
}

struct FxFinSmem {
    int32_t R[kBlock];             // each row's reference (largest chunk reference)
    unsigned long long T[kBlock];  // each row's total in row units
    int32_t rbad[kBlock];          // the row cannot be weighed
    unsigned long long qx;         // the removed draft's weight in its chunk
    unsigned long long tc;         // the draw's target inside its chunk
    unsigned long long wsum[kSWarpsPerCta];
    int32_t a, excl, kstar, tok;
    int32_t out[kBlock];  // the emitted tokens (fused: committed)
    int32_t flag[3];
};

// Request b is complete: decide the drafts, draw the token, write the
// outputs, rewind the counter (fused: commit the emitted tokens; a request
// whose rows cannot be weighed commits nothing and latches CLK_EINVAL).
// Block-wide.
template <int DT, bool FUSED>
__device__ __noinline__ void fx_finish(const SampleArgs& a, const LookupDev& Ldev, const unsigned long long* rec,
                                       int32_t b, FxFinSmem& fs, const FxPoly& poly)
{
    using E = SElem<DT>;
    const unsigned full = 0xFFFFFFFFu;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t L = a.len[b], NC = a.S, V = a.V;
    const float s = a.inv_temp[b] * kLog2e;
    const typename E::T* base = static_cast<const typename E::T*>(a.logits) + (int64_t)b * a.req_stride;
    const unsigned long long* rb = rec + (int64_t)b * kBlock * NC;
    __threadfence();
    // Each row's reference and total: 16 threads per row (row = tid / 16),
    // each taking the row's chunks sub, sub + 16, ..., then a butterfly over
    // the 16 (the same result in all of them).
    {
        const int32_t r = tid >> 4, sub = tid & 15;
        int32_t Rm = kFxNoRef, bad = 0;
        if (r < L) {
#pragma unroll 8
            for (int32_t k = sub; k < NC; k += 16) {
                const unsigned long long q = __ldcg(rb + (int64_t)r * NC + k);
                if (q == kFxBad) bad = 1;
                else Rm = max(Rm, fx_ref(q));
            }
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
            Rm = max(Rm, __shfl_xor_sync(full, Rm, o));
            bad |= __shfl_xor_sync(full, bad, o);
        }
        unsigned long long T = 0ull;
        if (r < L && !bad) {
#pragma unroll 8
            for (int32_t k = sub; k < NC; k += 16) {
                const unsigned long long q = __ldcg(rb + (int64_t)r * NC + k);
                T += fx_rowunits(fx_sum(q), Rm - fx_ref(q));
            }
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) T += __shfl_xor_sync(full, T, o);
        if (sub == 0 && r < L) {
            fs.R[r] = Rm;
            fs.T[r] = T;
            fs.rbad[r] = bad || Rm == kFxNoRef;
        }
    }
    __syncthreads();
    int32_t bad = 0;
    for (int32_t r = 0; r < L; ++r) bad |= fs.rbad[r];
    if (bad) {  // some row cannot be weighed: the empty result
        if (tid < kBlock) a.out_tok[(int64_t)b * kBlock + tid] = CLK_SENT;
        if (tid == 0) {
            a.accept[b] = 0;
            a.emitted[b] = 0;
            a.done[b] = 0u;
            if (FUSED) latch(Ldev.status, CLK_EINVAL, b);
        }
        __syncthreads();
        return;
    }
    // Every draft at once (lane r: row r's draft blk[r + 1]).
    if (warp == 0) {
        const bool has = lane < L - 1;
        const int32_t c = has ? a.block[(int64_t)b * kBlock + lane + 1] : CLK_SENT;
        const bool inv = c >= 0 && c < V;
        bool acc = false;
        unsigned long long qc = 0ull;
        if (has && inv) {
            const int32_t Rk = fx_ref(__ldcg(rb + (int64_t)lane * NC + c / kFxChunk));
            qc = fx_q1(E::value(base[(int64_t)lane * a.row_stride + c]), s, Rk, poly);
            const unsigned long long w = fx_rowunits(qc, fs.R[lane] - Rk);
            acc = fx_mulshift(fx_unit(a.uniform[((int64_t)b * kBlock + lane) * 2]), fs.T[lane]) < w;
        }
        const unsigned rej = __ballot_sync(full, has && !acc);
        const int32_t an = rej ? __ffs(rej) - 1 : L - 1;
        if (lane == an) {
            fs.a = an;
            fs.excl = (has && inv) ? c : -1;
            fs.qx = qc;
            fs.tok = CLK_SENT;
        }
    }
    __syncthreads();
    const int32_t ra = fs.a, excl = fs.excl;
    const unsigned long long* rr = rb + (int64_t)ra * NC;
    // The chunk of the draw, block-wide (thread j takes chunks j, j + 256,
    // ...): the chunks' totals with the removed draft taken out of its chunk
    // are summed for T', then scanned 256 chunks at a time to find the one
    // whose running total passes t = floor(k(u) T' / 2^24).
    {
        const int32_t Rr = fs.R[ra];
        const int32_t kx = excl >= 0 ? excl / kFxChunk : -1;
        const unsigned long long qx = fs.qx;
        auto tk = [&](int32_t k) -> unsigned long long {
            if (k >= NC) return 0ull;
            const unsigned long long q = __ldcg(rr + k);
            return fx_rowunits(fx_sum(q) - (k == kx ? qx : 0ull), Rr - fx_ref(q));
        };
        if (tid == 0) fs.kstar = -1;
        unsigned long long own = 0ull;
        for (int32_t k = tid; k < NC; k += kSThreads) own += tk(k);
        const unsigned long long total = fx_block_sum(own, fs.wsum);
        const unsigned long long t = fx_mulshift(fx_unit(a.uniform[((int64_t)b * kBlock + ra) * 2 + 1]), total);
        unsigned long long carry = 0ull;
        for (int32_t k0 = 0; k0 < NC; k0 += kSThreads) {
            const int32_t k = k0 + tid;
            const unsigned long long w = tk(k);
            unsigned long long slab;
            const unsigned long long incl = carry + fx_block_scan(w, fs.wsum, slab);
            if (w > 0ull && incl - w <= t && t < incl) {  // one chunk in all: the running totals partition [0, T')
                fs.kstar = k;
                fs.tc = fx_chunkunits(t - (incl - w), Rr - fx_ref(__ldcg(rr + k)));
            }
            carry += slab;
            __syncthreads();
            if (fs.kstar >= 0) break;
        }
    }
    // Inside the chunk: 4 consecutive entries per thread, a block-wide
    // exclusive scan of their sums, and the thread whose run holds the target
    // walks its 4 (c skipped: weight 0).
    const int32_t ks = fs.kstar;
    if (ks >= 0) {
        const int32_t Rk = fx_ref(__ldcg(rr + ks));
        const typename E::T* row = base + (int64_t)ra * a.row_stride;
        const int64_t v0 = (int64_t)ks * kFxChunk + 4 * tid;
        uint32_t q[4], own = 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t v = v0 + i;
            q[i] = (v < V && v != excl) ? fx_q1(E::value(row[v]), s, Rk, poly) : 0u;
            own += q[i];
        }
        unsigned long long chunk_total;
        const unsigned long long pre = fx_block_scan(own, fs.wsum, chunk_total) - own;
        const unsigned long long tc = fs.tc;
        if (pre <= tc && tc < pre + own) {  // one thread: the runs partition [0, chunk total)
            unsigned long long run = pre;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                run += q[i];
                if (run > tc) {
                    fs.tok = (int32_t)(v0 + i);
                    break;
                }
            }
        }
    }
    __syncthreads();
    if (tid < kBlock) {
        const int32_t r = tid;
        const int32_t out = r < ra ? a.block[(int64_t)b * kBlock + r + 1] : (r == ra ? fs.tok : CLK_SENT);
        a.out_tok[(int64_t)b * kBlock + r] = out;
        fs.out[r] = out;
    }
    if (tid == 0) {
        a.accept[b] = ra;
        a.emitted[b] = ra + 1;
        a.done[b] = 0u;
    }
    __syncthreads();
    if (FUSED) {
        const int32_t slot = a.slots[b];
        if (slot < 0 || slot >= Ldev.max_slots) {
            if (tid == 0) latch(Ldev.status, CLK_EINVAL, b);
        } else {
            block_commit_tokens(Ldev, slot, fs.out, ra + 1, fs.flag);
        }
        __syncthreads();
    }
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kSThreads, kFxCtas) k_sample_fx(SampleArgs a, FxPoly poly)
{
    extern __shared__ int32_t P[];  // B + 1
    __shared__ int32_t sm_warp[kSWarpsPerCta];
    __shared__ int32_t sm_last;
    __shared__ FxFinSmem fs;
    const int tid = threadIdx.x;
    const int32_t B = a.B;
    unsigned long long* rec = reinterpret_cast<unsigned long long*>(a.part);
    sample_prefix(a, P, sm_warp);
    // Requests with no rows (invalid length or temperature): empty result.
    if (blockIdx.x == 0) {
        for (int32_t b = tid; b < B; b += kSThreads) {
            if (sample_rows(a, b) != 0) continue;
            for (int r = 0; r < kBlock; ++r) a.out_tok[(int64_t)b * kBlock + r] = CLK_SENT;
            a.accept[b] = 0;
            a.emitted[b] = 0;
        }
    }
    const int64_t NC = a.S;
    const int64_t N = (int64_t)P[B] * NC;
    const int64_t lo = N * blockIdx.x / gridDim.x;
    const int64_t hi = N * (blockIdx.x + 1) / gridDim.x;
    int64_t k = lo;
    while (k < hi) {
        const int32_t b = sample_owner(P, B, k / NC);
        const int64_t k1 = min(hi, (int64_t)P[b + 1] * NC);
        fx_stream<DT, VEC>(a, P, b, 0, k, k1, poly, rec);
        __syncthreads();  // every warp's records are stored
        if (tid == 0) {
            __threadfence();
            const uint32_t n = (uint32_t)(k1 - k);
            const uint32_t need = (uint32_t)(P[b + 1] - P[b]) * (uint32_t)NC;
            sm_last = atomicAdd(a.done + b, n) + n == need;
        }
        __syncthreads();
        if (sm_last) fx_finish<DT, false>(a, LookupDev{}, rec, b, fs, poly);
        k = k1;
    }
}

// The sampler fused with the commit (clk_verify_sample_append), launched as
// a programmatic dependent of the proposal launch that produces the blocks
// and lengths.  As in the fused greedy verification, it first streams the
// segments of every request's predicted rows, max(1 + head, hint) (the
// short block when the hint is missing or not a valid length), while the
// proposal launch may still run; the counts of those segments are kept and
// decided after the wait, when the lengths are known.  Each CTA streams its
// even share of the predicted segments, waits, and then streams its share of
// the rows the prediction missed.  A request's total is max(predicted, L_b) rows of segments; the
// count that reaches it finishes the request (pairs of rows past L_b are
// never used).  A request with a valid temperature but an invalid length
// streams its predicted rows for nothing: the count that completes it only
// sets the counter back to zero.  The inverse temperatures are read before
// the wait, so they must not come from the proposal launch.
constexpr int kSMaxDefer = 32;
constexpr int64_t kSLateBytes = 90ll << 20;  // HBM bytes streamed before the late CTAs start (tuned)

// The block's next action, chosen by thread 0.
enum SampleAct : int32_t { kActStream, kActCheck, kActWait, kActDone };

struct SampleStepSmem {
    int64_t k, kend;          // the current phase's next segment and end (flat)
    int64_t kstop, hi1;       // where the first phase stopped; the end of this CTA's predicted share
    int64_t c0, c1;           // the piece to stream: segments [c0, c1) of request cb,
    int32_t cb, croff;        // rows counted from croff
    int32_t phase, act;
    int32_t db[kSMaxDefer];   // kept counts: request,
    uint32_t dc[kSMaxDefer];  // and the count its addition returned
    int32_t nd, ci;           // kept counts, and how many of them are decided
};

// The fused sampler's body, on the float weights (FX = false: per-warp
// (m, s) pairs per segment, sample_finish) or on the fixed-point ones
// (FX = true: units are 1024-entry chunks with one record each, fx_finish).
// Fin is the finisher's shared memory of the kind.
template <int DT, bool VEC, bool FX, typename Fin>
__device__ __forceinline__ void sample_step_body(const SampleArgs& a, const LookupDev& Ldev, const FxPoly& poly,
                                                 int32_t* sm_p, int32_t* sm_warp, Fin& fs, SampleStepSmem& ss)
{
    // sm_p: P1[B + 1] (predicted rows), P2[B + 1] (missed rows), then
    // Lc[B + 1] (after the wait: each request's length, read once)
    // Let the next launch (the next proposal) be scheduled; it waits for
    // this grid to complete before it reads anything this grid writes.  With
    // paired scratch halves only after this launch's own wait: the next
    // proposal may then let the next sampled verify start at once (on the
    // other half), and by then the verify before this one has completed.
    if (!a.paired) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x;
    const int32_t B = a.B;
    int32_t* P1 = sm_p;
    int32_t* P2 = sm_p + (B + 1);
    int32_t* Lc = sm_p + 2 * (B + 1);
    const int32_t base = min(kBlock, 1 + Ldev.p.head);
    rows_prefix(B, [&a, base](int32_t b) {
        if (!temp_valid(a.inv_temp[b])) return 0;
        const int32_t h = a.len_hint != nullptr ? a.len_hint[b] : 0;
        return len_valid(h) ? max(h, base) : base;
    }, P1, sm_warp);
    if (tid == 0) {
        // This CTA's share of the predicted segments.  As in the fused greedy
        // verification, the last `late` CTAs start only when the proposal
        // launch's CTAs leave their SMs, about kSLateBytes of HBM time in;
        // they get f8/8 of a share, less the shorter this launch.
        const int64_t n = (int64_t)P1[B] * a.S;
        const int64_t G = gridDim.x;
        const int64_t D = min((int64_t)a.late, G / 4);
        const int64_t bytes = (int64_t)P1[B] * a.V * (int64_t)sizeof(typename SElem<DT>::T);
        int64_t f8 = bytes > 0 ? 8 - (8 * kSLateBytes + bytes / 2) / bytes : 8;
        f8 = f8 < 0 ? 0 : (f8 > 8 ? 8 : f8);
        const int64_t Wtot = (G - D) * 8 + D * f8;
        auto start = [&](int64_t c) {  // n * W(c) / Wtot without overflow
            const int64_t w = c <= G - D ? c * 8 : (G - D) * 8 + (c - (G - D)) * f8;
            return (n / Wtot) * w + (n % Wtot) * w / Wtot;
        };
        const int64_t lo = start(blockIdx.x), hi = start(blockIdx.x + 1);
        ss.k = lo;
        ss.kend = hi;
        ss.hi1 = hi;
        ss.phase = 0;
        ss.nd = 0;
        ss.ci = 0;
    }
    // Phase 0: this CTA's predicted segments, counts kept (stopping early if
    // the list of kept counts is full); the wait; phase 1: its share of the
    // missed rows; phase 2: whatever phase 0 left.  After the wait every
    // kept count is decided: the one that equals its request's total
    // (max(predicted, L_b) rows of segments) finishes the request, or, for
    // an invalid length, only rewinds its counter.  The wait comes after the
    // whole predicted share: a request completes only once all of its
    // segments are read, so its finisher runs at the end whatever the order,
    // and a wait in the middle would pause every CTA at about the same time.
    for (;;) {
        if (tid == 0) {
            int32_t act = kActDone;
            for (;;) {
                if (ss.phase > 0 && ss.ci < ss.nd) {
                    act = kActCheck;
                    break;
                }
                if (ss.phase > 0) ss.ci = ss.nd = 0;
                if (ss.k < ss.kend && !(ss.phase == 0 && ss.nd == kSMaxDefer)) {
                    const int32_t* P = ss.phase == 1 ? P2 : P1;
                    const int32_t b = sample_owner(P, B, ss.k / a.S);
                    ss.cb = b;
                    ss.c0 = ss.k;
                    ss.c1 = min(ss.kend, (int64_t)P[b + 1] * a.S);
                    ss.croff = ss.phase == 1 ? P1[b + 1] - P1[b] : 0;
                    act = kActStream;
                    break;
                }
                if (ss.phase == 0) {
                    ss.kstop = ss.k;
                    act = kActWait;
                    break;
                }
                if (ss.phase == 1) {
                    ss.phase = 2;
                    ss.k = ss.kstop;
                    ss.kend = ss.hi1;
                    continue;
                }
                break;
            }
            ss.act = act;
        }
        __syncthreads();
        const int32_t act = ss.act;
        if (act == kActDone) break;
        if (act == kActStream) {
            const int32_t b = ss.cb;
            const int32_t* P = ss.phase == 1 ? P2 : P1;
            if constexpr (FX) {
                fx_stream<DT, VEC>(a, P, b, ss.croff, ss.c0, ss.c1, poly, reinterpret_cast<unsigned long long*>(a.part));
            } else {
                if (VEC) stream_vec<DT>(a, P, b, ss.croff, ss.c0, ss.c1);
                else stream_scalar<DT>(a, P, b, ss.croff, ss.c0, ss.c1);
            }
            __syncthreads();  // every warp's pairs (or chunk records) are stored
            if (tid == 0) {
                __threadfence();
                const uint32_t c = (uint32_t)(ss.c1 - ss.c0);
                ss.db[ss.nd] = b;
                ss.dc[ss.nd] = atomicAdd(a.done + b, c) + c;
                ss.nd += 1;
                ss.k = ss.c1;
            }
        } else if (act == kActCheck) {
            const int32_t b = ss.db[ss.ci];
            const int32_t Lb = Lc[b];
            const int32_t pr = P1[b + 1] - P1[b];
            const uint32_t total = (uint32_t)((pr > 0 && len_valid(Lb)) ? max(pr, Lb) : pr) * (uint32_t)a.S;
            if (ss.dc[ss.ci] == total) {
                if (len_valid(Lb)) {
                    if constexpr (FX) {
                        fx_finish<DT, true>(a, Ldev, reinterpret_cast<const unsigned long long*>(a.part), b, fs, poly);
                    } else {
                        sample_finish<DT, true>(a, Ldev, b, fs);
                    }
                } else if (tid == 0) {
                    a.done[b] = 0u;
                }
            }
            __syncthreads();
            if (tid == 0) ss.ci += 1;
        } else {  // kActWait
            asm volatile("griddepcontrol.wait;" ::: "memory");
            if (a.paired) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            rows_prefix(B, [&a, P1, Lc](int32_t b) {
                const int32_t pr = P1[b + 1] - P1[b];
                const int32_t Lb = __ldcg(a.len + b);
                Lc[b] = Lb;
                return (pr > 0 && len_valid(Lb)) ? max(0, Lb - pr) : 0;
            }, P2, sm_warp);
            // Requests with no rows (invalid length or temperature): the
            // empty result, nothing committed, an error.
            if (blockIdx.x == 0) {
                for (int32_t b = tid; b < B; b += kSThreads) {
                    if (sample_rows(a, b) != 0) continue;
                    for (int r = 0; r < kBlock; ++r) a.out_tok[(int64_t)b * kBlock + r] = CLK_SENT;
                    a.accept[b] = 0;
                    a.emitted[b] = 0;
                    latch(Ldev.status, CLK_EINVAL, b);
                }
            }
            if (tid == 0) {
                const int64_t n = (int64_t)P2[B] * a.S;
                ss.k = n * blockIdx.x / gridDim.x;
                ss.kend = n * (blockIdx.x + 1) / gridDim.x;
                ss.phase = 1;
            }
        }
        __syncthreads();
    }
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kSThreads, CLK_SAMPLE_CTAS) k_sample_step(SampleArgs a, LookupDev Ldev)
{
    extern __shared__ int32_t sm_p[];
    __shared__ int32_t sm_warp[kSWarpsPerCta];
    __shared__ FinSmem fs;
    __shared__ SampleStepSmem ss;
    sample_step_body<DT, VEC, false>(a, Ldev, FxPoly{}, sm_p, sm_warp, fs, ss);
}

// The exact sampler fused with the commit (clk_verify_sample_exact_append):
// the fused schedule above on 1024-entry chunks.
template <int DT, bool VEC>
__global__ void __launch_bounds__(kSThreads, kFxCtas) k_sample_step_fx(SampleArgs a, LookupDev Ldev, FxPoly poly)
{
    extern __shared__ int32_t sm_p[];
    __shared__ int32_t sm_warp[kSWarpsPerCta];
    __shared__ FxFinSmem fs;
    __shared__ SampleStepSmem ss;
    sample_step_body<DT, VEC, true>(a, Ldev, poly, sm_p, sm_warp, fs, ss);
}


int fx_sizes(int32_t dtype, int32_t V, int32_t B, int32_t* NC, size_t* bytes)
{
    if ((dtype != CLK_DTYPE_BF16 && dtype != CLK_DTYPE_F32) || V < 1 || V > kFxVMax || B < 0 || B > CLK_MAX_BATCH)
        return CLK_EINVAL;
    const int64_t nc = ((int64_t)V + kFxChunk - 1) / kFxChunk;
    *NC = (int32_t)nc;
    const size_t nb = (size_t)(B > 0 ? B : 1);
    *bytes = align_up(nb * sizeof(uint32_t), 16) + nb * kBlock * (size_t)nc * sizeof(unsigned long long);
    return CLK_OK;
}

// c_j = sqrt(2) (ln 2)^j / j! rounded to float, from the recurrence
// t_0 = sqrt(2), t_{j+1} = t_j ln2 / (j + 1) in double.
FxPoly fx_poly()
{
    FxPoly p;
    double t = 1.4142135623730951;
    const double ln2 = 0.6931471805599453;
    for (int j = 0; j < 7; ++j) {
        p.c[j] = (float)t;
        uint32_t bits;
        memcpy(&bits, &p.c[j], sizeof bits);
        p.c2[j] = ((unsigned long long)bits << 32) | bits;
        t = t * ln2 / (double)(j + 1);
    }
    return p;
}

template <int DT, bool VEC>
int launch_fx(const SampleArgs& a, cudaStream_t s)
{
    static std::atomic<int> cache[64];  // resident CTAs per SM, per device (calls from any host thread)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CLK_ECUDA;
    const size_t smem = (size_t)(a.B + 1) * sizeof(int32_t);
    auto kern = k_sample_fx<DT, VEC>;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return CLK_ECUDA;
    int occ = (dev >= 0 && dev < 64 && smem <= 4096) ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (occ <= 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kSThreads, smem <= 4096 ? 4096 : smem) !=
                cudaSuccess ||
            occ < 1)
            return CLK_ECUDA;
        if (dev >= 0 && dev < 64 && smem <= 4096) cache[dev].store(occ, std::memory_order_relaxed);
    }
    const int sms = num_sms();
    if (sms <= 0) return CLK_ECUDA;
    const int64_t chunks = (int64_t)a.B * kBlock * a.S;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((int64_t)occ * sms, chunks));
    kern<<<(unsigned)grid, kSThreads, smem, s>>>(a, fx_poly());
    return launch_status();
}

int sample_sizes(int32_t dtype, int32_t V, int32_t B, int32_t* S, size_t* bytes)
{
    if ((dtype != CLK_DTYPE_BF16 && dtype != CLK_DTYPE_F32) || V < 1 || B < 0 || B > CLK_MAX_BATCH)
        return CLK_EINVAL;
    const int64_t segs = ((int64_t)V + kSegElems - 1) / kSegElems;
    *S = (int32_t)segs;
    const size_t nb = (size_t)(B > 0 ? B : 1);
    *bytes = align_up(nb * sizeof(uint32_t), 16) + nb * kBlock * (size_t)segs * kSWarpsPerCta * sizeof(float2);
    return CLK_OK;
}

template <int DT, bool VEC, bool FUSED>
int launch_sample(const SampleArgs& a, const LookupDev& Ldev, cudaStream_t s)
{
    static std::atomic<int> cache[64];  // resident CTAs per SM, per device (calls from any host thread)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CLK_ECUDA;
    const size_t smem = (size_t)(FUSED ? 3 : 1) * (a.B + 1) * sizeof(int32_t);
    auto kern = FUSED ? k_sample_step<DT, VEC> : k_sample<DT, VEC>;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return CLK_ECUDA;
    int occ = (dev >= 0 && dev < 64 && smem <= 4096) ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (occ <= 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kSThreads, smem <= 4096 ? 4096 : smem) !=
                cudaSuccess ||
            occ < 1)
            return CLK_ECUDA;
        if (dev >= 0 && dev < 64 && smem <= 4096) cache[dev].store(occ, std::memory_order_relaxed);
    }
    const int sms = num_sms();
    if (sms <= 0) return CLK_ECUDA;
    const int64_t segs = (int64_t)a.B * kBlock * a.S;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((int64_t)occ * sms, segs));
    SampleArgs args = a;
    if (FUSED && a.late > 0) {
        // CTAs dispatched behind the proposal launch's CTAs: those beyond the
        // places the proposal leaves (as in the fused greedy verification).
        const int64_t taken = (int64_t)displaced_by_proposal<k_sample_step<DT, VEC>>(kSThreads, Ldev.nlev, occ) *
                              (a.B < sms ? a.B : sms);
        const int64_t late = grid - ((int64_t)occ * sms - taken);
        args.late = late > 0 ? (int32_t)late : 0;
    }
    if (!FUSED) {
        kern<<<(unsigned)grid, kSThreads, smem, s>>>(args, Ldev);
        return launch_status();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, kern, args, Ldev));
}

// The exact sampler fused with the commit: launched as launch_sample's fused
// path launches the float one (programmatic dependent of the proposal launch,
// the CTAs dispatched behind it given a smaller share).
template <int DT, bool VEC>
int launch_sample_fx_fused(const SampleArgs& a, const LookupDev& Ldev, cudaStream_t s)
{
    static std::atomic<int> cache[64];  // resident CTAs per SM, per device (calls from any host thread)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CLK_ECUDA;
    const size_t smem = (size_t)3 * (a.B + 1) * sizeof(int32_t);
    auto kern = k_sample_step_fx<DT, VEC>;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return CLK_ECUDA;
    int occ = (dev >= 0 && dev < 64 && smem <= 4096) ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (occ <= 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kSThreads, smem <= 4096 ? 4096 : smem) !=
                cudaSuccess ||
            occ < 1)
            return CLK_ECUDA;
        if (dev >= 0 && dev < 64 && smem <= 4096) cache[dev].store(occ, std::memory_order_relaxed);
    }
    const int sms = num_sms();
    if (sms <= 0) return CLK_ECUDA;
    const int64_t chunks = (int64_t)a.B * kBlock * a.S;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((int64_t)occ * sms, chunks));
    SampleArgs args = a;
    if (a.late > 0) {
        const int64_t taken = (int64_t)displaced_by_proposal<k_sample_step_fx<DT, VEC>>(kSThreads, Ldev.nlev, occ) *
                              (a.B < sms ? a.B : sms);
        const int64_t late = grid - ((int64_t)occ * sms - taken);
        args.late = late > 0 ? (int32_t)late : 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, kern, args, Ldev, fx_poly()));
}

}  // namespace
}  // namespace clk

using namespace clk;

extern "C" int clk_verify_sample_scratch_bytes(int32_t dtype, int32_t V, int32_t B, size_t* bytes)
{
    if (bytes == nullptr) return CLK_EINVAL;
    int32_t S = 0;
    return sample_sizes(dtype, V, B, &S, bytes);
}

extern "C" int clk_verify_sample_exact_scratch_bytes(int32_t dtype, int32_t V, int32_t B, size_t* bytes)
{
    if (bytes == nullptr) return CLK_EINVAL;
    int32_t NC = 0;
    return fx_sizes(dtype, V, B, &NC, bytes);
}

namespace {

// Checks and launches both entry points; h == nullptr: stateless.
int sample_entry(clk_lookup* h, const int32_t* d_slots, const void* d_logits, int32_t dtype, int64_t row_stride,
                 int64_t req_stride, int32_t V, int32_t B, const int32_t* d_block, const int32_t* d_len,
                 const int32_t* d_len_hint, const float* d_inv_temp, const float* d_uniform, int32_t* d_accept, int32_t* d_emitted,
                 int32_t* d_out_tok, void* d_scratch, size_t scratch_bytes, cudaStream_t cs, bool paired = false,
                 bool exact = false)
{
    int32_t S = 0;
    size_t need = 0;
    int rc = exact ? fx_sizes(dtype, V, B, &S, &need) : sample_sizes(dtype, V, B, &S, &need);
    if (rc != CLK_OK) return rc;
    if (h != nullptr) {
        rc = check_batch(h, B);
        if (rc != CLK_OK) return rc;
        if (!ok_i32(d_slots)) return CLK_EINVAL;
    }
    if (row_stride < V || req_stride < 0 || (B > 1 && req_stride < row_stride)) return CLK_EINVAL;
    const size_t esz = dtype == CLK_DTYPE_BF16 ? 2 : 4;
    if (d_logits == nullptr || !aligned(d_logits, esz)) return CLK_EINVAL;
    if (!ok_i32(d_block) || !ok_i32(d_len) || !ok_i32(d_accept) || !ok_i32(d_emitted) || !ok_i32(d_out_tok) ||
        d_inv_temp == nullptr || !aligned(d_inv_temp, 4) || d_uniform == nullptr || !aligned(d_uniform, 4))
        return CLK_EINVAL;
    if (d_scratch == nullptr || !aligned(d_scratch, 16) || scratch_bytes < need) return CLK_EINVAL;
    if (d_len_hint != nullptr && !aligned(d_len_hint, 4)) return CLK_EINVAL;
    if (B == 0) return CLK_OK;
    SampleArgs a;
    a.logits = d_logits;
    a.row_stride = row_stride;
    a.req_stride = req_stride;
    a.V = V;
    a.B = B;
    a.S = S;
    a.block = d_block;
    a.len = d_len;
    a.len_hint = d_len_hint;
    a.inv_temp = d_inv_temp;
    a.uniform = d_uniform;
    a.accept = d_accept;
    a.emitted = d_emitted;
    a.out_tok = d_out_tok;
    a.done = static_cast<uint32_t*>(d_scratch);
    a.part = reinterpret_cast<float2*>(static_cast<char*>(d_scratch) + align_up((size_t)B * sizeof(uint32_t), 16));
    a.slots = d_slots;
    // Fused: it may overlap the proposal launch before it; the count of its
    // CTAs that start behind that launch is worked out at launch.
    a.late = h != nullptr && !h->alone ? 1 : 0;
    a.paired = paired ? 1 : 0;
    const int64_t W = 16 / (int64_t)esz;
    const bool vec = aligned(d_logits, 16) && V % W == 0 && row_stride % W == 0 && req_stride % W == 0;
    const bool bf = dtype == CLK_DTYPE_BF16;
    if (exact && h != nullptr) {
        const LookupDev& L = h->dev;
        if (bf) return vec ? launch_sample_fx_fused<CLK_DTYPE_BF16, true>(a, L, cs)
                           : launch_sample_fx_fused<CLK_DTYPE_BF16, false>(a, L, cs);
        return vec ? launch_sample_fx_fused<CLK_DTYPE_F32, true>(a, L, cs)
                   : launch_sample_fx_fused<CLK_DTYPE_F32, false>(a, L, cs);
    }
    if (exact) {
        if (bf) return vec ? launch_fx<CLK_DTYPE_BF16, true>(a, cs) : launch_fx<CLK_DTYPE_BF16, false>(a, cs);
        return vec ? launch_fx<CLK_DTYPE_F32, true>(a, cs) : launch_fx<CLK_DTYPE_F32, false>(a, cs);
    }
    if (h != nullptr) {
        const LookupDev& L = h->dev;
        if (bf) return vec ? launch_sample<CLK_DTYPE_BF16, true, true>(a, L, cs)
                           : launch_sample<CLK_DTYPE_BF16, false, true>(a, L, cs);
        return vec ? launch_sample<CLK_DTYPE_F32, true, true>(a, L, cs)
                   : launch_sample<CLK_DTYPE_F32, false, true>(a, L, cs);
    }
    const LookupDev none = {};
    if (bf) return vec ? launch_sample<CLK_DTYPE_BF16, true, false>(a, none, cs)
                       : launch_sample<CLK_DTYPE_BF16, false, false>(a, none, cs);
    return vec ? launch_sample<CLK_DTYPE_F32, true, false>(a, none, cs)
               : launch_sample<CLK_DTYPE_F32, false, false>(a, none, cs);
}

}  // namespace

extern "C" int clk_verify_sample(const void* d_logits, int32_t dtype, int64_t row_stride, int64_t req_stride,
                                 int32_t V, int32_t B, const int32_t* d_block, const int32_t* d_len,
                                 const float* d_inv_temp, const float* d_uniform, int32_t* d_accept,
                                 int32_t* d_emitted, int32_t* d_out_tok, void* d_scratch, size_t scratch_bytes,
                                 clk_stream_t s)
{
    return sample_entry(nullptr, nullptr, d_logits, dtype, row_stride, req_stride, V, B, d_block, d_len, nullptr,
                        d_inv_temp, d_uniform, d_accept, d_emitted, d_out_tok, d_scratch, scratch_bytes,
                        (cudaStream_t)s);
}

extern "C" int clk_verify_sample_exact(const void* d_logits, int32_t dtype, int64_t row_stride, int64_t req_stride,
                                       int32_t V, int32_t B, const int32_t* d_block, const int32_t* d_len,
                                       const float* d_inv_temp, const float* d_uniform, int32_t* d_accept,
                                       int32_t* d_emitted, int32_t* d_out_tok, void* d_scratch, size_t scratch_bytes,
                                       clk_stream_t s)
{
    return sample_entry(nullptr, nullptr, d_logits, dtype, row_stride, req_stride, V, B, d_block, d_len, nullptr,
                        d_inv_temp, d_uniform, d_accept, d_emitted, d_out_tok, d_scratch, scratch_bytes,
                        (cudaStream_t)s, false, true);
}

namespace {

// The fused sampled verification, float (exact = false) or fixed-point
// weights.  A scratch of two halves (each half of the buffer, rounded down to
// 256 bytes, whatever the batch, and each at least what this batch needs):
// consecutive calls alternate them, and the next proposal may let the next
// call start streaming before its own wait.  One buffer: the next proposal
// must not let the next verify start before this one completes.
int sample_append(clk_lookup* h, const int32_t* d_slots, const void* d_logits, int32_t dtype, int64_t row_stride,
                  int64_t req_stride, int32_t V, int32_t B, const int32_t* d_block, const int32_t* d_len,
                  const int32_t* d_len_hint, const float* d_inv_temp, const float* d_uniform, int32_t* d_accept,
                  int32_t* d_emitted, int32_t* d_out_tok, void* d_scratch, size_t scratch_bytes, clk_stream_t s,
                  bool exact)
{
    if (h == nullptr) return CLK_EINVAL;
    int32_t S = 0;
    size_t need = 0;
    const size_t half_bytes = (scratch_bytes / 2) & ~(size_t)255;
    const int sz = exact ? fx_sizes(dtype, V, B, &S, &need) : sample_sizes(dtype, V, B, &S, &need);
    const bool paired = sz == CLK_OK && d_scratch != nullptr && half_bytes >= need;
    void* half = paired ? static_cast<char*>(d_scratch) + (size_t)h->sparity * half_bytes : d_scratch;
    const int rc = sample_entry(h, d_slots, d_logits, dtype, row_stride, req_stride, V, B, d_block, d_len,
                                d_len_hint, d_inv_temp, d_uniform, d_accept, d_emitted, d_out_tok, half,
                                paired ? half_bytes : scratch_bytes, (cudaStream_t)s, paired, exact);
    if (rc == CLK_OK && paired) {
        h->sparity ^= 1;
        h->last_fused = kFusedSampledPaired;
        h->vsince = 1;
    } else {
        h->last_fused = rc == CLK_OK ? kFusedSampled : kFusedNone;
    }
    return rc;
}

}  // namespace

extern "C" int clk_verify_sample_append(clk_lookup* h, const int32_t* d_slots, const void* d_logits, int32_t dtype,
                                        int64_t row_stride, int64_t req_stride, int32_t V, int32_t B,
                                        const int32_t* d_block, const int32_t* d_len, const int32_t* d_len_hint,
                                        const float* d_inv_temp, const float* d_uniform, int32_t* d_accept,
                                        int32_t* d_emitted, int32_t* d_out_tok, void* d_scratch,
                                        size_t scratch_bytes, clk_stream_t s)
{
    return sample_append(h, d_slots, d_logits, dtype, row_stride, req_stride, V, B, d_block, d_len, d_len_hint,
                         d_inv_temp, d_uniform, d_accept, d_emitted, d_out_tok, d_scratch, scratch_bytes, s, false);
}

extern "C" int clk_verify_sample_exact_append(clk_lookup* h, const int32_t* d_slots, const void* d_logits,
                                              int32_t dtype, int64_t row_stride, int64_t req_stride, int32_t V,
                                              int32_t B, const int32_t* d_block, const int32_t* d_len,
                                              const int32_t* d_len_hint, const float* d_inv_temp,
                                              const float* d_uniform, int32_t* d_accept, int32_t* d_emitted,
                                              int32_t* d_out_tok, void* d_scratch, size_t scratch_bytes,
                                              clk_stream_t s)
{
    return sample_append(h, d_slots, d_logits, dtype, row_stride, req_stride, V, B, d_block, d_len, d_len_hint,
                         d_inv_temp, d_uniform, d_accept, d_emitted, d_out_tok, d_scratch, scratch_bytes, s, true);
}
