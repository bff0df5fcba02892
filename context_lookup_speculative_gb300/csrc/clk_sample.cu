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
// flat list of (request, row, segment) triples.  Each thread keeps a running
// maximum m and sum s = sum exp(x t - m) over its strided vectors of a
// segment; each warp combines its 32 threads' pairs with shuffles in a fixed
// order and stores one (m, s) pair per segment and warp in the scratch, so no
// barrier is needed per segment.  When a CTA leaves a request it adds the
// number of that request's segments it finished to the request's counter;
// the CTA that completes the count finishes the request: it combines the
// pairs of each row in a fixed order, decides all acceptances at once, finds
// the segment that holds the sample from the pairs and the token inside it by
// reading that one segment again.  Every reduction has a fixed order, so the
// results do not depend on the grid or on timing.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "clk.h"
#include "clk_device.cuh"
#include "clk_host.h"

namespace clk {
namespace {

constexpr int kSThreads = 256;
constexpr int kSWarpsPerCta = kSThreads / 32;
constexpr int kSUnroll = 4;
constexpr int64_t kSegElems = 16384;  // elements per segment

struct SampleArgs {
    const void* logits;
    int64_t row_stride;  // elements
    int64_t req_stride;  // elements
    int32_t V;
    int32_t B;
    int32_t S;            // segments per row
    const int32_t* block;
    const int32_t* len;
    const float* inv_temp;  // [B]
    const float* uniform;   // [B][16][2]
    int32_t* accept;
    int32_t* emitted;
    int32_t* out_tok;
    uint32_t* done;  // [B] segments finished per request
    float2* part;    // [B][16][S][kSWarpsPerCta] (m, s) per warp
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
    __device__ static void unpack(const uint4& v, float* f)
    {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
};

// Running (max, sum of exp(y - max)) of a set of values y.
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
    return MS{m, a.s * __expf(a.m - m) + b.s * __expf(b.m - m)};
}

// Adds W values y_i = x_i * t.
template <int W>
__device__ __forceinline__ void ms_add(MS& r, const float* x, float t)
{
    float y[W];
    float vm = -INFINITY;
#pragma unroll
    for (int i = 0; i < W; ++i) {
        y[i] = x[i] * t;
        vm = fmaxf(vm, y[i]);
    }
    if (vm > r.m) {
        r.s = r.s == 0.0f ? 0.0f : r.s * __expf(r.m - vm);
        r.m = vm;
    }
    if (r.m == -INFINITY) return;  // every value so far is -inf: weight 0
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < W; ++i) acc += __expf(y[i] - r.m);
    r.s += acc;
}

// Warp-wide merge in a fixed (butterfly) order; every lane gets the result.
__device__ __forceinline__ MS ms_warp(MS r)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        MS q;
        q.m = __shfl_xor_sync(0xFFFFFFFFu, r.m, o);
        q.s = __shfl_xor_sync(0xFFFFFFFFu, r.s, o);
        // the lower lane's pair first, so both lanes compute the same value
        r = (threadIdx.x & o) ? ms_merge(q, r) : ms_merge(r, q);
    }
    return r;
}

// Adds one value y = x * t.
__device__ __forceinline__ void ms_add1(MS& r, float x, float t)
{
    const float y = x * t;
    if (y > r.m) {
        r.s = r.s == 0.0f ? 0.0f : r.s * __expf(r.m - y);
        r.m = y;
    }
    if (r.m != -INFINITY) r.s += __expf(y - r.m);
}

// P[b] = rows of requests b' < b; P[B] = total.  Block-wide.
__device__ __forceinline__ void sample_prefix(const SampleArgs& a, int32_t* P, int32_t* sm_warp)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t B = a.B;
    const int32_t per = (B + kSThreads - 1) / kSThreads;
    const int32_t b0 = min(B, tid * per), b1 = min(B, b0 + per);
    int32_t local = 0;
    for (int32_t b = b0; b < b1; ++b) local += sample_rows(a, b);
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
        P[b] = run;
        run += sample_rows(a, b);
    }
    if (tid == kSThreads - 1) P[B] = sm_warp[kSWarpsPerCta - 1];
    __syncthreads();
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
__device__ __forceinline__ void seg_range(const SampleArgs& a, const int32_t* P, int32_t b, int64_t k,
                                          const char*& row, int32_t& u0, int32_t& u1, int32_t& r, int32_t& sg)
{
    using E = SElem<DT>;
    constexpr int W = VEC ? E::W : 1;
    const int64_t ri = k / a.S;
    sg = (int32_t)(k - ri * a.S);
    r = (int32_t)(ri - P[b]);
    row = static_cast<const char*>(a.logits) +
          ((int64_t)b * a.req_stride + (int64_t)r * a.row_stride) * (int64_t)sizeof(typename E::T);
    const int64_t e0 = (int64_t)sg * kSegElems, e1 = min(e0 + kSegElems, (int64_t)a.V);
    u0 = (int32_t)(e0 / W);
    u1 = (int32_t)(e1 / W);
}

// Streams segments [k0, k1) of request b and stores one (m, s) pair per
// segment and warp.  Vector path: two groups of kSUnroll 16-byte loads per
// thread alternate, and the next segment's first group is issued before the
// current segment's last group is reduced.
template <int DT>
__device__ __forceinline__ void stream_vec(const SampleArgs& a, const int32_t* P, int32_t b, int64_t k0, int64_t k1)
{
    using E = SElem<DT>;
    constexpr int W = E::W;
    constexpr int32_t G = kSUnroll * kSThreads;  // vectors per group
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float t = a.inv_temp[b];
    const char* rowp;
    int32_t u0, u1, r, sg;
    seg_range<DT, true>(a, P, b, k0, rowp, u0, u1, r, sg);
    const uint4* row = reinterpret_cast<const uint4*>(rowp);
    int32_t gb = u0 + tid;
    int64_t k = k0;
    MS run = ms_empty();
    uint4 X[kSUnroll], Y[kSUnroll];
    auto load = [&](const uint4* rw, int32_t base, int32_t end, uint4* d) {
#pragma unroll
        for (int u = 0; u < kSUnroll; ++u) {
            const int32_t vi = base + u * kSThreads;
            if (vi < end) d[u] = __ldcs(rw + vi);
        }
    };
    auto reduce = [&](const uint4* d, int32_t base, int32_t end) {
#pragma unroll
        for (int u = 0; u < kSUnroll; ++u) {
            const int32_t vi = base + u * kSThreads;
            if (vi < end) {
                float f[W];
                E::unpack(d[u], f);
                ms_add<W>(run, f, t);
            }
        }
    };
    // One half-step: the group in C is current; the next group goes into N.
    auto half = [&](uint4* C, uint4* N) -> bool {
        const uint4* nrow = row;
        int32_t nu1 = u1, ngb = gb + G, nr = r, nsg = sg;
        bool more = true, seg_end = false;
        if (gb - tid + G >= u1) {
            seg_end = true;
            if (k + 1 < k1) {
                int32_t nu0;
                seg_range<DT, true>(a, P, b, k + 1, rowp, nu0, nu1, nr, nsg);
                nrow = reinterpret_cast<const uint4*>(rowp);
                ngb = nu0 + tid;
            } else {
                more = false;
            }
        }
        if (more) load(nrow, ngb, nu1, N);
        reduce(C, gb, u1);
        if (seg_end) {
            const MS w = ms_warp(run);
            if (lane == 0) part_of(a, b, r, sg)[warp] = make_float2(w.m, w.s);
            run = ms_empty();
            ++k;
        }
        row = nrow;
        u1 = nu1;
        gb = ngb;
        r = nr;
        sg = nsg;
        return more;
    };
    load(row, gb, u1, X);
    for (;;) {
        if (!half(X, Y)) break;
        if (!half(Y, X)) break;
    }
}

// Scalar path (rows not 16-byte aligned): one segment at a time.
template <int DT>
__device__ __forceinline__ void stream_scalar(const SampleArgs& a, const int32_t* P, int32_t b, int64_t k0,
                                              int64_t k1)
{
    using E = SElem<DT>;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float t = a.inv_temp[b];
    for (int64_t k = k0; k < k1; ++k) {
        const char* rowp;
        int32_t u0, u1, r, sg;
        seg_range<DT, false>(a, P, b, k, rowp, u0, u1, r, sg);
        const typename E::T* row = reinterpret_cast<const typename E::T*>(rowp);
        MS run = ms_empty();
        for (int32_t i = u0 + tid; i < u1; i += kSThreads) ms_add1(run, E::value(row[i]), t);
        const MS w = ms_warp(run);
        if (lane == 0) part_of(a, b, r, sg)[warp] = make_float2(w.m, w.s);
    }
}

struct FinSmem {
    float m[kBlock], s[kBlock];  // each row's combined pair
    float ex;                    // weight exp(x_c t - m) of the removed draft
    float tgt;                   // the sample's target inside the chosen segment
    int32_t a, excl, seg, tok;
    float wsum[kSWarpsPerCta];
};

// Request b is complete (all of its segments' pairs are stored): decide the
// drafts, draw the token, write the outputs, rewind the counter.  Block-wide.
template <int DT>
__device__ __forceinline__ void sample_finish(const SampleArgs& a, int32_t b, FinSmem& fs)
{
    using E = SElem<DT>;
    const unsigned full = 0xFFFFFFFFu;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t L = a.len[b], S = a.S, V = a.V;
    const float t = a.inv_temp[b];
    const typename E::T* base = static_cast<const typename E::T*>(a.logits) + (int64_t)b * a.req_stride;
    __threadfence();
    // Each row's pair: the segments' pairs in index order, then the butterfly.
    for (int32_t r = warp; r < L; r += kSWarpsPerCta) {
        const float2* pp = part_of(a, b, r, 0);
        MS acc = ms_empty();
        for (int32_t i = lane; i < S * kSWarpsPerCta; i += 32) {
            const float2 q = __ldcg(pp + i);
            acc = ms_merge(acc, MS{q.x, q.y});
        }
        acc = ms_warp(acc);
        if (lane == 0) {
            fs.m[r] = acc.m;
            fs.s[r] = acc.s;
        }
    }
    __syncthreads();
    // Acceptance of every draft at once (lane r: row r's draft blk[r + 1]).
    if (warp == 0) {
        const bool has = lane < L - 1;
        const int32_t c = has ? a.block[(int64_t)b * kBlock + lane + 1] : CLK_SENT;
        const bool inv = c >= 0 && c < V;
        float ec = 0.0f;
        if (has && inv) ec = __expf(E::value(base[(int64_t)lane * a.row_stride + c]) * t - fs.m[lane]);
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
    // The segment holding the sample: running sum of the segments' weights
    // (relative to the row's maximum, the removed draft taken out of its
    // segment) against u * (row sum - removed weight).
    if (warp == 0) {
        const float target = a.uniform[((int64_t)b * kBlock + ra) * 2 + 1] * fmaxf(0.0f, fs.s[ra] - fs.ex);
        const float2* pp = part_of(a, b, ra, 0);
        const int32_t exseg = excl >= 0 ? (int32_t)(excl / kSegElems) : -1;
        float carry = 0.0f;
        int32_t found = -1, lastpos = -1;
        float before = 0.0f;
        for (int32_t k0 = 0; k0 < S && found < 0; k0 += 32) {
            const int32_t k = k0 + lane;
            float w = 0.0f;
            if (k < S) {
                for (int i = 0; i < kSWarpsPerCta; ++i) {
                    const float2 q = __ldcg(pp + (int64_t)k * kSWarpsPerCta + i);
                    if (q.y > 0.0f) w += q.y * __expf(q.x - mra);
                }
                if (k == exseg) w = fmaxf(0.0f, w - fs.ex);
            }
            float incl = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(full, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned cross = __ballot_sync(full, k < S && carry + incl > target);
            const unsigned pos = __ballot_sync(full, k < S && w > 0.0f);
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
            fs.tgt = found >= 0 ? target - before : INFINITY;  // no crossing: the last positive weight
        }
    }
    __syncthreads();
    // Inside the segment: each thread a contiguous run of the segment's
    // elements; block-wide exclusive scan of the runs' sums; the first thread
    // whose run crosses the target walks its run.
    constexpr int32_t kRun = (int32_t)(kSegElems / kSThreads);
    const int32_t sg = fs.seg;
    const typename E::T* row = base + (int64_t)ra * a.row_stride;
    const int64_t v0 = sg < 0 ? 0 : (int64_t)sg * kSegElems + (int64_t)tid * kRun;
    const int64_t v1 = sg < 0 ? 0 : min(v0 + kRun, min((int64_t)(sg + 1) * kSegElems, (int64_t)V));
    float own = 0.0f;
    int64_t lastv = -1;
    for (int64_t v = v0; v < v1; ++v) {
        if (v == excl) continue;
        const float e = __expf(E::value(row[v]) * t - mra);
        own += e;
        if (e > 0.0f) lastv = v;
    }
    float incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(full, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) fs.wsum[warp] = incl;
    if (tid == 0) fs.tok = CLK_SENT;
    __syncthreads();
    float pre = incl - own;
    for (int w = 0; w < warp; ++w) pre += fs.wsum[w];
    const float tgt = fs.tgt;
    const bool crosses = own > 0.0f && pre + own > tgt && !(pre > tgt);
    if (crosses) {
        float run = pre;
        int64_t tok = lastv;
        for (int64_t v = v0; v < v1; ++v) {
            if (v == excl) continue;
            run += __expf(E::value(row[v]) * t - mra);
            if (run > tgt) {
                tok = v;
                break;
            }
        }
        fs.tok = (int32_t)tok;  // exactly one thread crosses
    }
    __syncthreads();
    if (fs.tok == CLK_SENT) {
        // no crossing (rounding, or the target past the segment): the
        // segment's last element of positive weight
        const unsigned has = __ballot_sync(full, lastv >= 0);
        if (has && lane == 31 - __clz(has)) fs.wsum[warp] = __int_as_float((int32_t)lastv);
        else if (lane == 0 && !has) fs.wsum[warp] = __int_as_float(-1);
        __syncthreads();
        if (tid == 0) {
            for (int w = kSWarpsPerCta - 1; w >= 0; --w) {
                const int32_t v = __float_as_int(fs.wsum[w]);
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
    }
    if (tid == 0) {
        a.accept[b] = fs.a;
        a.emitted[b] = fs.a + 1;
        a.done[b] = 0u;
    }
    __syncthreads();
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kSThreads, 4) k_sample(SampleArgs a)
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
        if (VEC) stream_vec<DT>(a, P, b, k, k1);
        else stream_scalar<DT>(a, P, b, k, k1);
        __syncthreads();  // every warp's pairs are stored
        if (tid == 0) {
            __threadfence();
            const uint32_t n = (uint32_t)(k1 - k);
            const uint32_t need = (uint32_t)(P[b + 1] - P[b]) * (uint32_t)S;
            sm_last = atomicAdd(a.done + b, n) + n == need;
        }
        __syncthreads();
        if (sm_last) sample_finish<DT>(a, b, fs);
        k = k1;
    }
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

template <int DT, bool VEC>
int launch_sample(const SampleArgs& a, cudaStream_t s)
{
    static int cache[64] = {0};  // resident CTAs per SM, per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CLK_ECUDA;
    const size_t smem = (size_t)(a.B + 1) * sizeof(int32_t);
    auto kern = k_sample<DT, VEC>;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return CLK_ECUDA;
    int occ = (dev >= 0 && dev < 64 && smem <= 4096) ? cache[dev] : 0;
    if (occ <= 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kSThreads, smem <= 4096 ? 4096 : smem) !=
                cudaSuccess ||
            occ < 1)
            return CLK_ECUDA;
        if (dev >= 0 && dev < 64 && smem <= 4096) cache[dev] = occ;
    }
    const int sms = num_sms();
    if (sms <= 0) return CLK_ECUDA;
    const int64_t segs = (int64_t)a.B * kBlock * a.S;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((int64_t)occ * sms, segs));
    kern<<<(unsigned)grid, kSThreads, smem, s>>>(a);
    return launch_status();
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

extern "C" int clk_verify_sample(const void* d_logits, int32_t dtype, int64_t row_stride, int64_t req_stride,
                                 int32_t V, int32_t B, const int32_t* d_block, const int32_t* d_len,
                                 const float* d_inv_temp, const float* d_uniform, int32_t* d_accept,
                                 int32_t* d_emitted, int32_t* d_out_tok, void* d_scratch, size_t scratch_bytes,
                                 clk_stream_t s)
{
    int32_t S = 0;
    size_t need = 0;
    int rc = sample_sizes(dtype, V, B, &S, &need);
    if (rc != CLK_OK) return rc;
    if (row_stride < V || req_stride < 0 || (B > 1 && req_stride < row_stride)) return CLK_EINVAL;
    const size_t esz = dtype == CLK_DTYPE_BF16 ? 2 : 4;
    if (d_logits == nullptr || !aligned(d_logits, esz)) return CLK_EINVAL;
    if (!ok_i32(d_block) || !ok_i32(d_len) || !ok_i32(d_accept) || !ok_i32(d_emitted) || !ok_i32(d_out_tok) ||
        d_inv_temp == nullptr || !aligned(d_inv_temp, 4) || d_uniform == nullptr || !aligned(d_uniform, 4))
        return CLK_EINVAL;
    if (d_scratch == nullptr || !aligned(d_scratch, 16) || scratch_bytes < need) return CLK_EINVAL;
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
    a.inv_temp = d_inv_temp;
    a.uniform = d_uniform;
    a.accept = d_accept;
    a.emitted = d_emitted;
    a.out_tok = d_out_tok;
    a.done = static_cast<uint32_t*>(d_scratch);
    a.part = reinterpret_cast<float2*>(static_cast<char*>(d_scratch) + align_up((size_t)B * sizeof(uint32_t), 16));
    const int64_t W = 16 / (int64_t)esz;
    const bool vec = aligned(d_logits, 16) && V % W == 0 && row_stride % W == 0 && req_stride % W == 0;
    cudaStream_t cs = (cudaStream_t)s;
    if (dtype == CLK_DTYPE_BF16)
        return vec ? launch_sample<CLK_DTYPE_BF16, true>(a, cs) : launch_sample<CLK_DTYPE_BF16, false>(a, cs);
    return vec ? launch_sample<CLK_DTYPE_F32, true>(a, cs) : launch_sample<CLK_DTYPE_F32, false>(a, cs);
}
