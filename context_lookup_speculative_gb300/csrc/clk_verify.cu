// Greedy verification (HyperQwen context-lookup article, "三步走", last
// paragraph; the Polish page's "the first rejected proposal ends the run"):
// row-wise argmax over the target logits of each verify block, fused with the
// accepted-prefix count, the emitted tokens and (clk_verify_append) the
// commit of those tokens into the request's history (the next proposal
// launch indexes them).
//
// Layout of the work: the rows that must be read (L_b rows of request b) are
// numbered 0..R-1 in request order and seen as one flat range of R * V/W
// 16-byte vectors (W elements each).  A grid of G CTAs, G = SMs x resident
// CTAs, splits that range evenly; each CTA streams its contiguous share with
// 128-bit loads (up to 8 in flight per thread), reduces every row piece it covers
// to a packed (order-preserving value bits << 32 | ~index) 64-bit key, and
// merges it into the row's key with one atomicMax (max value, then lowest
// index; independent of CTA order).  Each CTA then adds the vectors it
// covered to the request's counter; the CTA that completes a request (its
// add reaches L_b * V/W) reads the row keys and finishes that request:
// argmax tokens, accepted count, emitted tokens and, fused, the token commit.
// No CTA waits on another.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "clk.h"
#include "clk_device.cuh"
#include "clk_host.h"

namespace clk {

constexpr int kVThreads = 256;
constexpr int kVWarps = kVThreads / 32;
constexpr int kUnroll = 4;

struct VerifyArgs {
    const void* logits;
    int64_t row_stride;
    int64_t req_stride;
    int32_t V;
    int32_t B;
    const int32_t* block;
    const int32_t* len;
    const int32_t* len_hint;  // fused: predicted block lengths (may be null)
    int32_t* argmax;
    int32_t* accept;
    int32_t* emitted;
    int32_t* out_tok;
    unsigned long long* keys;  // [B * 16]
    unsigned long long* done;  // [B]
    const int32_t* slots;      // fused only
    int32_t late;              // fused: trailing CTAs that start behind the proposal launch (0: none)
    int32_t aligned;           // fused: split few rows in whole-row parts (latency-bound launches)
};

// Order-preserving 32-bit key of a float: larger value, larger key; +0 == -0.
__device__ __forceinline__ uint32_t ord_key(float f)
{
    uint32_t u = __float_as_uint(f);
    if (f == 0.0f) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned long long pack_key(uint32_t key, uint32_t idx)
{
    return ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}

constexpr uint32_t kNanKey = 0xFFFFFFFFu;  // any NaN beats every number

__device__ __forceinline__ bool len_ok(int32_t l) { return l >= 1 && l <= kBlock; }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t hmax2_nan_u32(uint32_t a, uint32_t b)
{
    __nv_bfloat162 x, y;
    memcpy(&x, &a, 4);
    memcpy(&y, &b, 4);
    const __nv_bfloat162 m = __hmax2_nan(x, y);
    uint32_t r;
    memcpy(&r, &m, 4);
    return r;
}

template <int DT>
struct Elem;
template <>
struct Elem<CLK_DTYPE_BF16> {
    using T = uint16_t;
    static constexpr int W = 8;
    __device__ static float value(T x) { return __uint_as_float((uint32_t)x << 16); }
    __device__ static void unpack(const uint4& v, float* f)
    {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    }
    // Max of the 8 values by packed bf16x2 max that propagates NaN; any NaN of
    // the vector sets bit 15 or 31 of `nanacc` (then the max value is unused).
    __device__ static float vec_max(const uint4& v, uint32_t& nanacc)
    {
        const uint32_t m2 = hmax2_nan_u32(hmax2_nan_u32(v.x, v.y), hmax2_nan_u32(v.z, v.w));
        nanacc |= (m2 & 0x7FFF7FFFu) + 0x007F007Fu;
        return fmaxf(bf16_lo(m2), bf16_hi(m2));
    }
    static constexpr uint32_t kNanMask = 0x80008000u;
};
template <>
struct Elem<CLK_DTYPE_F32> {
    using T = float;
    static constexpr int W = 4;
    __device__ static float value(T x) { return x; }
    __device__ static void unpack(const uint4& v, float* f)
    {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
    __device__ static float vec_max(const uint4& v, uint32_t& nanacc)
    {
        const uint32_t m = 0x7FFFFFFFu, c = 0x007FFFFFu;
        nanacc |= ((v.x & m) + c) | ((v.y & m) + c) | ((v.z & m) + c) | ((v.w & m) + c);
        return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                     fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
    static constexpr uint32_t kNanMask = 0x80000000u;
};

__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }

// Loads vectors base + u * kVThreads (u < U) that lie below v1.
// Vector indices inside a row fit in 32 bits (V < 2^31).
template <int U>
__device__ __forceinline__ void load_group(const uint4* row, int32_t base, int32_t v1, uint4* x)
{
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int32_t vi = base + u * kVThreads;
        if (vi < v1) x[u] = ld_stream(row + vi);
    }
}

template <int DT, int U>
__device__ __forceinline__ void reduce_group(const uint4* x, int32_t base, int32_t v1, float& best, int32_t& bvi,
                                             uint4& bvec, uint32_t& nanacc)
{
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int32_t vi = base + u * kVThreads;
        if (vi < v1) {
            const float m = Elem<DT>::vec_max(x[u], nanacc);
            if (m > best) {
                best = m;
                bvi = vi;
                bvec = x[u];
            }
        }
    }
}

// This thread's packed key over vectors [v0, v1) of a row (vector path).
// Two register groups of U vectors alternate: the next group's loads are
// issued before the current group is reduced, so up to 2 x U 16-byte loads
// per thread are in flight.  The index inside the winning vector is
// recovered from the vector kept in registers.
template <int DT, int U = kUnroll>
__device__ __forceinline__ unsigned long long scan_vec(const void* row_ptr, int32_t v0, int32_t v1)
{
    using E = Elem<DT>;
    constexpr int W = E::W;
    constexpr int32_t S = U * kVThreads;
    const uint4* row = reinterpret_cast<const uint4*>(row_ptr);
    const int32_t first = v0 + (int32_t)threadIdx.x;
    if (first >= v1) return 0ull;
    float best = -__int_as_float(0x7F800000);  // -inf
    int32_t bvi = -1;
    uint4 bvec = make_uint4(0u, 0u, 0u, 0u);
    uint32_t nanacc = 0u;
    uint4 a[U], b[U];
    load_group<U>(row, first, v1, a);
    for (int32_t base = first; base < v1; base += 2 * S) {
        load_group<U>(row, base + S, v1, b);
        reduce_group<DT, U>(a, base, v1, best, bvi, bvec, nanacc);
        if (base + S >= v1) break;
        load_group<U>(row, base + 2 * S, v1, a);
        reduce_group<DT, U>(b, base + S, v1, best, bvi, bvec, nanacc);
    }
    if (nanacc & E::kNanMask) {
        // Rare path: the first NaN of this thread's elements.
        for (int32_t vi = first; vi < v1; vi += kVThreads) {
            float f[W];
            E::unpack(row[vi], f);
#pragma unroll
            for (int e = 0; e < W; ++e)
                if (f[e] != f[e]) return pack_key(kNanKey, (uint32_t)vi * W + e);
        }
    }
    if (bvi < 0) return pack_key(ord_key(best), (uint32_t)first * W);  // every element is -inf
    float f[W];
    E::unpack(bvec, f);
    int e0 = W - 1;
#pragma unroll
    for (int e = W - 1; e >= 0; --e)
        if (f[e] == best) e0 = e;
    return pack_key(ord_key(best), (uint32_t)bvi * W + e0);
}

// This thread's packed key over elements [v0, v1) of a row (unaligned rows).
template <int DT>
__device__ __forceinline__ unsigned long long scan_scalar(const void* row_ptr, int64_t v0, int64_t v1)
{
    using E = Elem<DT>;
    const typename E::T* row = reinterpret_cast<const typename E::T*>(row_ptr);
    const int64_t first = v0 + threadIdx.x;
    if (first >= v1) return 0ull;
    float best = -__int_as_float(0x7F800000);
    int64_t bi = first;
    for (int64_t i = first; i < v1; i += kVThreads) {
        const float f = E::value(row[i]);
        if (f != f) return pack_key(kNanKey, (uint32_t)i);
        if (f > best) {
            best = f;
            bi = i;
        }
    }
    return pack_key(ord_key(best), (uint32_t)bi);
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

// Max over the block; the result is valid in thread 0.
__device__ __forceinline__ unsigned long long block_max_u64(unsigned long long v, unsigned long long* sm_red)
{
    v = warp_max_u64(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) sm_red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < kVWarps ? sm_red[lane] : 0ull;
        v = warp_max_u64(v);
    }
    return v;
}

// Rows of request b past the first `base` rows: max(0, L_b - base) for a
// valid length 1 <= L_b <= 16, else 0.
__device__ __forceinline__ int32_t rows_after(int32_t l, int32_t base) { return len_ok(l) ? max(0, l - base) : 0; }

// P[b] = rows(b') summed over requests b' < b; P[B] = total.  Block-wide.
template <typename Rows>
__device__ __forceinline__ void block_prefix(int32_t B, Rows rows, int32_t* P, int32_t* sm_warp)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t per = (B + kVThreads - 1) / kVThreads;
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
        int32_t s = lane < kVWarps ? sm_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < kVWarps) sm_warp[lane] = s;  // inclusive warp totals
    }
    __syncthreads();
    int32_t run = (incl - local) + (warp > 0 ? sm_warp[warp - 1] : 0);
    for (int32_t b = b0; b < b1; ++b) {
        const int32_t r = P[b];
        P[b] = run;
        run += r;
    }
    if (tid == kVThreads - 1) P[B] = sm_warp[kVWarps - 1];
    __syncthreads();
}

__device__ __forceinline__ void named_barrier(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// block_prefix computed by warps 1 .. kVWarps-1 only (named barrier 1), so
// that warp 0 can do other work meanwhile.  Called by those warps only.
template <typename Rows>
__device__ __forceinline__ void rest_prefix(int32_t B, Rows rows, int32_t* P, int32_t* sm_warp)
{
    constexpr int kW = kVWarps - 1, kT = kW * 32;
    const int t = threadIdx.x - 32, lane = t & 31, w = t >> 5;
    const int32_t per = (B + kT - 1) / kT;
    const int32_t b0 = min(B, t * per), b1 = min(B, b0 + per);
    int32_t local = 0;
    for (int32_t b = b0; b < b1; ++b) {  // rows(b) read once, kept in P[b] (as in block_prefix)
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
    if (lane == 31) sm_warp[w] = incl;
    named_barrier(1, kT);
    if (w == 0) {
        int32_t v = lane < kW ? sm_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, v, o);
            if (lane >= o) v += y;
        }
        if (lane < kW) sm_warp[lane] = v;  // inclusive warp totals
    }
    named_barrier(1, kT);
    int32_t run = (incl - local) + (w > 0 ? sm_warp[w - 1] : 0);
    for (int32_t b = b0; b < b1; ++b) {
        const int32_t r = P[b];
        P[b] = run;
        run += r;
    }
    if (t == kT - 1) P[B] = sm_warp[kW - 1];
}

// P[b] = rows_after(L_b', base) summed over requests b' < b; P[B] = total.
__device__ __forceinline__ void block_row_prefix(const int32_t* __restrict__ len, int32_t B, int32_t base, int32_t* P,
                                                 int32_t* sm_warp)
{
    block_prefix(B, [len, base](int32_t b) { return rows_after(len[b], base); }, P, sm_warp);
}

struct VerifySmem {
    unsigned long long red[kVWarps];
    int32_t warp[kVWarps];
    int32_t last;
    int32_t slot;  // fused: the slot of the request a count may finish
};

// One row piece: this CTA's maximum over vectors [s0, s1) of row r of
// request b, merged into the row's key.
template <int DT, bool VEC, int U = kUnroll>
__device__ __forceinline__ void piece_max(const VerifyArgs& a, int32_t b, int32_t r, int64_t s0, int64_t s1,
                                          VerifySmem& sm)
{
    using T = typename Elem<DT>::T;
    const char* row = static_cast<const char*>(a.logits) +
                      ((int64_t)b * a.req_stride + (int64_t)r * a.row_stride) * (int64_t)sizeof(T);
    unsigned long long key = VEC ? scan_vec<DT, U>(row, (int32_t)s0, (int32_t)s1) : scan_scalar<DT>(row, s0, s1);
    key = block_max_u64(key, sm.red);
    if (threadIdx.x == 0) atomicMax(a.keys + (int64_t)b * kBlock + r, key);
}

// Request b is complete: argmax tokens, accepted count, emitted tokens; the
// row keys and the counter go back to zero; fused, the tokens are committed
// to slot `slot` (its history, the ring of its last tokens, its length and
// counters).  Lb outside 1..16 gives the empty result.  Run by warp 0; the
// row keys, the drafts and the slot's length and last block length arrive
// in one round trip, and the commit is stores only.
// Counter addition with release (this CTA's key merges before it) and acquire
// (the merges of every CTA whose addition came before, for the finisher).
__device__ __forceinline__ unsigned long long atom_add_acq_rel(unsigned long long* p, unsigned long long v)
{
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}

// Loads issued as written (volatile): a finisher's loads are issued before
// the barriers that follow them and consumed after.
__device__ __forceinline__ unsigned long long ld_cg_u64(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.global.cg.u64 %0, [%1];" : "=l"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ int32_t ld_cg_i32(const int32_t* p)
{
    int32_t v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// What a finisher reads, one value per lane of warp 0: lane r < 16 the key
// of row r and the draft blk[r + 1]; lane 16 the slot's history length and
// lane 17 its last block length (fused).
struct FinLoads {
    unsigned long long kv;
    int32_t nxt;
    int32_t sv;
};

template <bool FUSED>
__device__ __forceinline__ FinLoads finalize_loads(const VerifyArgs& a, const LookupDev& L, int32_t b, int32_t slot)
{
    const int lane = threadIdx.x & 31;
    FinLoads f;
    f.kv = lane < kBlock ? ld_cg_u64(a.keys + (int64_t)b * kBlock + lane) : 0ull;
    f.nxt = (lane + 1 < kBlock) ? ld_cg_i32(a.block + (int64_t)b * kBlock + lane + 1) : CLK_SENT;
    f.sv = 0;
    const bool sok = FUSED && slot >= 0 && slot < L.max_slots;
    if (sok && lane == 16) f.sv = ld_cg_i32(&L.state[slot].n);
    if (sok && lane == 17) f.sv = ld_cg_i32(&L.state[slot].cur_len);
    return f;
}

template <bool FUSED>
__device__ __forceinline__ void finalize(const VerifyArgs& a, const LookupDev& L, int32_t b, int32_t Lb,
                                         int32_t slot, bool have = false, FinLoads pre = FinLoads{0ull, CLK_SENT, 0})
{
    if (threadIdx.x >= 32) return;
    const unsigned full = 0xFFFFFFFFu;
    const int lane = threadIdx.x;
    const FinLoads f = have ? pre : finalize_loads<FUSED>(a, L, b, slot);
    const bool valid = len_ok(Lb);
    unsigned long long* kp = a.keys + (int64_t)b * kBlock;
    const unsigned long long kv = f.kv;
    const int32_t nxt = f.nxt;
    const bool sok = FUSED && slot >= 0 && slot < L.max_slots;
    const int32_t sv = f.sv;
    const int32_t g = (valid && lane < Lb) ? (int32_t)(0xFFFFFFFFu - (uint32_t)kv) : CLK_SENT;
    const unsigned match = __ballot_sync(full, valid && lane < Lb - 1 && nxt == g);
    const int32_t acc = __ffs(~match) - 1;
    const int32_t out = (valid && lane <= acc) ? g : CLK_SENT;
    if (lane < kBlock) {
        a.argmax[(int64_t)b * kBlock + lane] = g;
        a.out_tok[(int64_t)b * kBlock + lane] = out;
        kp[lane] = 0ull;
    }
    if (lane == 0) {
        a.accept[b] = valid ? acc : 0;
        a.emitted[b] = valid ? acc + 1 : 0;
        a.done[b] = 0ull;
    }
    if (!FUSED) return;
    const int32_t n = __shfl_sync(full, sv, 16);
    const int32_t cur_len = __shfl_sync(full, sv, 17);
    if (!valid || !sok) {
        if (lane == 0) latch(L.status, CLK_EINVAL, b);
        return;
    }
    // The commit of clk_lookup_append: count = acc + 1 <= 16 tokens.
    const int32_t count = acc + 1;
    const unsigned bad_tok = __ballot_sync(full, lane < count && !token_ok(L, out));
    if ((int64_t)n + count > L.cap || bad_tok) {
        if (lane == 0) latch(L.status, bad_tok && (int64_t)n + count <= L.cap ? CLK_EINVAL : CLK_ECAPACITY, slot);
        return;
    }
    SlotState* st = L.state + slot;
    if (lane < count) {
        hist_of(L, slot)[n + lane] = out;
        st->ring[(n + lane) & (kRing - 1)] = out;
    }
    if (lane == 0) {
        st->n = n + count;
        st->cur_len = 0;
        if (cur_len != 0) {
            // No other CTA touches this slot in the launch: additions whose
            // result nothing waits for.
            atomicAdd(reinterpret_cast<unsigned long long*>(&st->accepted), (unsigned long long)(count - 1));
            atomicAdd(reinterpret_cast<unsigned long long*>(&st->emitted), (unsigned long long)count);
            const int cls = (L.p.tail > 0 && cur_len == long_len(L.p)) ? 1 : 0;
            atomicAdd(reinterpret_cast<unsigned long long*>(&st->accept_hist[cls][count - 1]), 1ull);
        }
    }
}

// Adds `add` verified vectors to request b; the CTA whose addition reaches
// `need` finishes the request.  Block-wide.
template <bool FUSED>
__device__ __forceinline__ void piece_count(const VerifyArgs& a, const LookupDev& L, int32_t b, unsigned long long add,
                                            unsigned long long need, int32_t Lb, VerifySmem& sm)
{
    if (threadIdx.x == 0) {
        const unsigned long long c = atom_add_acq_rel(a.done + b, add) + add;
        const int32_t slot = FUSED ? a.slots[b] : -1;  // loaded in the same round trip
        sm.last = c == need ? 1 : 0;
        sm.slot = slot;
    }
    __syncthreads();
    if (sm.last) finalize<FUSED>(a, L, b, Lb, sm.slot);
    __syncthreads();
}

// Largest b with P[b] <= ri.
__device__ __forceinline__ int32_t owner_of(const int32_t* P, int32_t B, int64_t ri)
{
    int32_t b = 0, top = B;
    while (b < top) {
        const int32_t mid = (b + top + 1) >> 1;
        if (P[mid] <= ri) b = mid; else top = mid - 1;
    }
    return b;
}

// Verification of the rows counted by the prefix P (rows past `base` of each
// request) split evenly over the grid; `need_rows(b)` is the total number of
// rows request b reads in this launch.
template <int DT, bool VEC, bool FUSED, typename NeedRows>
__device__ __forceinline__ void verify_rows(const VerifyArgs& a, const LookupDev& L, const int32_t* P, int32_t base,
                                            int64_t vpr, NeedRows need_rows, VerifySmem& sm)
{
    const int32_t B = a.B;
    const int64_t total = (int64_t)P[B] * vpr;
    int64_t lo = total * blockIdx.x / gridDim.x;
    const int64_t hi = total * (blockIdx.x + 1) / gridDim.x;
    if (lo >= hi) return;
    int64_t ri = lo / vpr;
    int32_t b = owner_of(P, B, ri);
    while (lo < hi) {
        while (P[b + 1] <= ri) ++b;
        const int32_t r = base + (int32_t)(ri - P[b]);
        const int64_t s0 = lo - ri * vpr;
        const int64_t s1 = min(hi, (ri + 1) * vpr) - ri * vpr;
        piece_max<DT, VEC>(a, b, r, s0, s1, sm);
        const int32_t Lb = a.len[b];
        piece_count<FUSED>(a, L, b, (unsigned long long)(s1 - s0),
                           (unsigned long long)need_rows(b, Lb) * (unsigned long long)vpr, Lb, sm);
        ri += 1;
        lo = ri * vpr;
    }
}

// Stateless verification (clk_verify_greedy): the block lengths are inputs,
// so the rows to read are known at launch.
template <int DT, bool VEC>
__global__ void __launch_bounds__(kVThreads, 4) k_verify(VerifyArgs a, LookupDev L)
{
    extern __shared__ int32_t sm_prefix[];  // B + 1
    __shared__ VerifySmem sm;
    const int32_t B = a.B;
    block_row_prefix(a.len, B, 0, sm_prefix, sm.warp);
    // Requests with no rows to read get their outputs here.
    if (blockIdx.x == 0) {
        for (int32_t b = threadIdx.x; b < B; b += kVThreads) {
            if (len_ok(a.len[b])) continue;
            for (int r = 0; r < kBlock; ++r) {
                a.argmax[(int64_t)b * kBlock + r] = CLK_SENT;
                a.out_tok[(int64_t)b * kBlock + r] = CLK_SENT;
            }
            a.accept[b] = 0;
            a.emitted[b] = 0;
        }
    }
    const int64_t vpr = VEC ? (int64_t)a.V / Elem<DT>::W : (int64_t)a.V;
    verify_rows<DT, VEC, false>(a, L, sm_prefix, 0, vpr, [](int32_t, int32_t l) { return l; }, sm);
}

// Verification fused with the commit (clk_verify_append), launched as a
// programmatic dependent of the proposal launch that produces the blocks and
// lengths.  Before it waits for that launch it reads, for every request, the
// rows of a predicted length (the short block, or the caller's hint, e.g. the
// previous step's length, when that is longer); after the wait it also reads
// the rows the prediction missed.  Every addition to a request's vector
// counter returns the new count; a count that equals the request's total
// (known only after the wait, max(predicted, true length) rows) finishes the
// request, so additions made before the wait are checked after it.  The
// answer does not depend on the prediction; a wrong one costs only reads.
//
// Each CTA streams its even share of the predicted rows in two halves.
// Between them it waits for the proposal launch (done by then in the steady
// state, where this launch overlaps it), checks the counts it deferred, lays
// out the missed rows and streams its share of them; the second half of the
// predicted rows follows with every count checked at once.  The latency-
// bound work (the checks, the missed rows' short pieces) thus runs while the
// other CTAs stream, and the launch ends soon after its last bytes arrive.
// A CTA with a short share (small batches) streams all of it first.
constexpr int kVMaxDefer = 32;
constexpr int64_t kVSplitMin = 64 * kVThreads;  // vectors: shares below this are not split
constexpr int64_t kLateBytes = 120ll << 20;     // HBM bytes streamed before the late CTAs start (tuned)
constexpr int64_t kVSmallBytes = 32ll << 20;     // logits (16 rows a request) of a latency-bound launch
constexpr int kVSmallPerSm = 2;                  // its CTAs per SM

// Rows read before the wait for request b.
__device__ __forceinline__ int32_t predicted_rows(const VerifyArgs& a, int32_t b, int32_t base)
{
    const int32_t h = a.len_hint != nullptr ? a.len_hint[b] : 0;
    return len_ok(h) ? max(h, base) : base;
}

struct StepSmem {
    int32_t db[kVMaxDefer];             // deferred checks: request,
    unsigned long long dc[kVMaxDefer];  // the count its addition returned,
    int32_t ds[kVMaxDefer];             // and its slot
    int32_t nd;
    int32_t waited;
    int32_t acc_b;               // the request whose vectors this CTA has
    unsigned long long acc_add;  // merged but not yet counted, and how many
};

template <int DT, bool VEC>
__global__ void __launch_bounds__(kVThreads, 4) k_verify_step(VerifyArgs a, LookupDev L)
{
    // P1[B + 1] (predicted rows), P2[B + 1] (missed rows), then Lc[B + 1]
    // (after the wait: each request's length, read once)
    extern __shared__ int32_t sm_prefix[];
    __shared__ VerifySmem sm;
    __shared__ StepSmem ss;
    const int tid = threadIdx.x;
    const int32_t B = a.B;
    int32_t* P1 = sm_prefix;
    int32_t* P2 = sm_prefix + (B + 1);
    int32_t* Lc = sm_prefix + 2 * (B + 1);
    const int32_t base = min(kBlock, 1 + L.p.head);
    const int64_t vpr = VEC ? (int64_t)a.V / Elem<DT>::W : (int64_t)a.V;
    if (tid == 0) {
        ss.nd = 0;
        ss.waited = 0;
        ss.acc_b = -1;
        ss.acc_add = 0ull;
    }
    block_prefix(B, [&a, base](int32_t b) { return predicted_rows(a, b, base); }, P1, sm.warp);

    // Vectors read for request b: its predicted rows, or its true length
    // when that is longer (valid lengths only).
    auto total = [&](int32_t b, int32_t Lb) -> unsigned long long {
        const int32_t pr = P1[b + 1] - P1[b];
        return (unsigned long long)(len_ok(Lb) ? max(Lb, pr) : pr) * (unsigned long long)vpr;
    };
    // Thread 0: count the vectors of request b that this CTA merged (one
    // addition per request and run of pieces; release for the merges,
    // acquire for the finisher) and keep the count it returned, with the
    // slot, for the check (made once the lengths are known).
    auto defer = [&](int32_t b, unsigned long long add) {
        const unsigned long long c = atom_add_acq_rel(a.done + b, add) + add;
        const int32_t slot = a.slots[b];  // the same round trip
        const int32_t i = ss.nd;
        ss.db[i] = b;
        ss.dc[i] = c;
        ss.ds[i] = slot;
        ss.nd = i + 1;
    };
    // Block-wide: count what is still pending; the first call waits for the
    // proposal launch and lays out the missed rows in P2; then decide the
    // deferred counts.
    auto flush = [&]() {
        // (uniform: these were last written before a barrier)
        if (ss.waited && ss.acc_b < 0 && ss.nd == 0) return;
        if (tid == 0 && ss.acc_b >= 0) {
            defer(ss.acc_b, ss.acc_add);
            ss.acc_b = -1;
            ss.acc_add = 0ull;
        }
        __syncthreads();
        if (!ss.waited) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            // Only now let the next launch (the next proposal) be scheduled:
            // the proposal after it may then start the next fused verify at
            // once, and by now the previous verify, which used the same half
            // of the scratch as that one, has completed.  The next proposal
            // waits for this grid before it reads anything this grid writes.
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            if (tid < 32) {
                // A count that reached the request's predicted vectors
                // finishes it whenever its length is within the prediction
                // (the common case): warp 0 reads that length with the
                // finisher's loads, in one round trip, and finishes at once,
                // while the other warps lay out the missed rows.
                int32_t spec = -1;
                for (int32_t i = 0; i < ss.nd; ++i) {
                    const int32_t b = ss.db[i];
                    if (ss.dc[i] == (unsigned long long)(P1[b + 1] - P1[b]) * (unsigned long long)vpr) spec = i;
                }
                if (spec >= 0) {
                    const int32_t b = ss.db[spec];
                    const FinLoads pre = finalize_loads<true>(a, L, b, ss.ds[spec]);
                    const int32_t Lb = ld_cg_i32(a.len + b);
                    if (ss.dc[spec] == total(b, Lb)) {
                        finalize<true>(a, L, b, Lb, ss.ds[spec], true, pre);
                        if (tid == 0) ss.dc[spec] = 0ull;  // decided: no later check matches it
                    }
                }
            } else {
                rest_prefix(B, [&a, P1, Lc](int32_t b) {
                    const int32_t Lb = __ldcg(a.len + b);
                    Lc[b] = Lb;
                    return len_ok(Lb) ? max(0, Lb - (P1[b + 1] - P1[b])) : 0;
                }, P2, sm.warp);
            }
            if (tid == 0) ss.waited = 1;
            __syncthreads();
        }
        // The finisher is warp 0 alone: the remaining checks need no barrier.
        if (tid < 32) {
            const int32_t nd = ss.nd;
            for (int32_t i = 0; i < nd; ++i) {
                const int32_t b = ss.db[i];
                if (ss.dc[i] == total(b, Lc[b])) finalize<true>(a, L, b, Lc[b], ss.ds[i]);
            }
            __syncwarp();
            if (tid == 0) ss.nd = 0;
        }
        __syncthreads();
    };
    // Vectors [from, to) of the flat range laid out by prefix P (row r of
    // request b at position P[b] + r - row0), rows row0 + ... of each
    // request, piece by piece (one piece per row).  A CTA counts once per
    // run of pieces of the same request: before the wait the count is
    // deferred (checked once the lengths are known); after it the count is
    // checked at once.
    auto stream = [&](const int32_t* P, bool missed, int64_t from, int64_t to) {
        if (from >= to) return;
        int64_t ri = from / vpr;
        int32_t b = owner_of(P, B, ri);
        int64_t lo = from;
        while (lo < to) {
            while (P[b + 1] <= ri) ++b;
            const int64_t s0 = lo - ri * vpr;
            const int64_t s1 = min(to, (ri + 1) * vpr) - ri * vpr;
            const int32_t row0 = missed ? P1[b + 1] - P1[b] : 0;
            piece_max<DT, VEC>(a, b, row0 + (int32_t)(ri - P[b]), s0, s1, sm);
            if (tid == 0) {
                if (b != ss.acc_b) {
                    if (ss.acc_b >= 0) defer(ss.acc_b, ss.acc_add);
                    ss.acc_b = b;
                    ss.acc_add = 0ull;
                }
                ss.acc_add += (unsigned long long)(s1 - s0);
            }
            __syncthreads();
            if (ss.waited ? ss.nd > 0 : ss.nd >= kVMaxDefer - 1) flush();
            ri += 1;
            lo = ri * vpr;
        }
    };

    // The predicted rows' flat range, split over the grid.  In the fused
    // step the proposal launch's CTAs still hold registers when this launch
    // starts, so its last `late` CTAs (dispatched last) start only when they
    // leave, about kLateBytes of HBM time in.  Those CTAs get f8/8 of a
    // share, less the shorter this launch; the split still covers the range
    // exactly, so only the timing depends on it.
    const int64_t total1 = (int64_t)P1[B] * vpr;
    const int64_t G = gridDim.x;
    const int64_t D = min((int64_t)a.late, G / 4);
    const int64_t bytes1 = total1 * (int64_t)(VEC ? 16 : sizeof(typename Elem<DT>::T));
    int64_t f8 = bytes1 > 0 ? 8 - (8 * kLateBytes + bytes1 / 2) / bytes1 : 8;
    f8 = f8 < 0 ? 0 : (f8 > 8 ? 8 : f8);
    const int64_t Wtot = (G - D) * 8 + D * f8;
    auto start = [&](int64_t c) {  // total1 * W(c) / Wtot without overflow
        const int64_t w = c <= G - D ? c * 8 : (G - D) * 8 + (c - (G - D)) * f8;
        return (total1 / Wtot) * w + (total1 % Wtot) * w / Wtot;
    };
    int64_t lo = start(blockIdx.x);
    int64_t hi = start(blockIdx.x + 1);
    if (a.aligned && P1[B] > 0 && P1[B] <= G - D && 3 * (int64_t)P1[B] > G - D) {
        // Rows about as many as the CTAs (a latency-bound launch with short
        // rows): one or two equal parts of a row per CTA (the first ones), so
        // that no CTA's share crosses a row boundary, where its loads would
        // drain and restart.  (With many parts a row, few shares cross one.)
        const int64_t R1 = P1[B], m = (G - D) / R1, c = blockIdx.x;
        lo = hi = 0;
        if (c < R1 * m) {
            const int64_t row = c / m, part = c % m;
            lo = row * vpr + vpr * part / m;
            hi = row * vpr + vpr * (part + 1) / m;
        }
    }
    const int64_t mid = (hi - lo >= kVSplitMin) ? lo + (hi - lo) / 2 : hi;
    stream(P1, false, lo, mid);
    flush();
    // This CTA's share of the rows the prediction missed.
    const int64_t total2 = (int64_t)P2[B] * vpr;
    stream(P2, true, total2 * blockIdx.x / gridDim.x, total2 * (blockIdx.x + 1) / gridDim.x);
    flush();
    stream(P1, false, mid, hi);
    flush();
}

// Resident CTAs per SM of kernel `Kern` and the SM count, packed as
// occ * 1024 + sms; cached per kernel and device for small shared memory.
template <auto Kern>
int occupancy(size_t smem, int* packed)
{
    constexpr int kDevices = 64;
    // One table per kernel (template argument).  Calls may come from several
    // host threads: the entries are atomic (any thread may fill an entry;
    // they all compute the same value).
    static std::atomic<int> cache[kDevices];
    const auto kern = Kern;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CLK_ECUDA;
    const bool cacheable = dev >= 0 && dev < kDevices && smem <= 4096;
    if (cacheable) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) {
            *packed = c;
            return CLK_OK;
        }
    }
    int occ = 0;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return CLK_ECUDA;
    // Sized for 4 KB so that the cached value holds for every cacheable size.
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kVThreads, cacheable ? 4096 : smem) !=
            cudaSuccess ||
        occ < 1)
        return CLK_ECUDA;
    const int sms = num_sms();
    if (sms <= 0 || sms >= 1024) return CLK_ECUDA;
    *packed = occ * 1024 + sms;
    if (cacheable) cache[dev].store(*packed, std::memory_order_relaxed);
    return CLK_OK;
}

template <auto Kern>
int verify_grid(size_t smem, int32_t B, int64_t vpr, int64_t* grid_out)
{
    int packed = 0;
    const int rc = occupancy<Kern>(smem, &packed);
    if (rc != CLK_OK) return rc;
    const int occ = packed / 1024, sms = packed % 1024;
    const int64_t max_work = (int64_t)B * kBlock * vpr;
    int64_t grid = (max_work + 4 * kVThreads - 1) / (4 * kVThreads);
    grid = grid < 1 ? 1 : grid;
    if (grid > (int64_t)occ * sms) grid = (int64_t)occ * sms;
    *grid_out = grid;
    return CLK_OK;
}

// Launches the fused step with at most `per_sm_cap` CTAs per SM (0: as many
// as fit).
template <int DT, bool VEC>
int launch_step(const VerifyArgs& a, const LookupDev& L, size_t smem, int64_t vpr, int per_sm_cap, cudaStream_t s)
{
    auto kern = k_verify_step<DT, VEC>;
    int64_t grid = 0;
    int rc = verify_grid<k_verify_step<DT, VEC>>(smem, a.B, vpr, &grid);
    if (rc != CLK_OK) return rc;
    int packed = 0;
    rc = occupancy<k_verify_step<DT, VEC>>(smem, &packed);
    if (rc != CLK_OK) return rc;
    const int occ = packed / 1024, sms = packed % 1024;
    if (per_sm_cap > 0 && grid > (int64_t)per_sm_cap * sms) grid = (int64_t)per_sm_cap * sms;
    VerifyArgs args = a;
    args.aligned = per_sm_cap > 0 ? 1 : 0;
    if (a.late > 0) {
        // a.late > 0: the call follows a proposal launch it may overlap.  The
        // proposal's CTAs (one a request, on min(B, SMs) SMs) each take the
        // place of some CTAs of this launch; the CTAs beyond the places left
        // (dispatched last) start only when the proposal's leave.
        const int64_t taken = (int64_t)displaced_by_proposal<k_verify_step<DT, VEC>>(kVThreads, L.nlev, occ) *
                              (a.B < sms ? a.B : sms);
        const int64_t late = grid - ((int64_t)occ * sms - taken);
        args.late = late > 0 ? (int32_t)late : 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kVThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, kern, args, L));
}

template <int DT, bool VEC, bool FUSED>
int launch_verify(const VerifyArgs& a, const LookupDev& L, cudaStream_t s)
{
    constexpr int W = VEC ? Elem<DT>::W : 1;
    const int64_t vpr = (int64_t)a.V / W;
    const size_t smem = (size_t)(FUSED ? 3 : 1) * (a.B + 1) * sizeof(int32_t);
    int64_t grid = 0;
    if (!FUSED) {
        auto kern = k_verify<DT, VEC>;
        int rc = verify_grid<k_verify<DT, VEC>>(smem, a.B, vpr, &grid);
        if (rc != CLK_OK) return rc;
        kern<<<(unsigned)grid, kVThreads, smem, s>>>(a, L);
        return launch_status();
    }
    // A launch whose logits are few (at most kVSmallBytes for all 16 rows of
    // every request) is latency-bound.  It keeps to two CTAs per SM, so that
    // the next step's proposal finds room beside it, and splits few rows in
    // whole-row parts.
    const int64_t max_bytes = (int64_t)a.B * kBlock * vpr * (int64_t)(VEC ? 16 : sizeof(typename Elem<DT>::T));
    return launch_step<DT, VEC>(a, L, smem, vpr, max_bytes <= kVSmallBytes ? kVSmallPerSm : 0, s);
}

int verify_dispatch(const VerifyArgs& a, int32_t dtype, bool fused, const LookupDev& L, cudaStream_t s)
{
    const int64_t esz = dtype == CLK_DTYPE_BF16 ? 2 : 4;
    const int64_t W = 16 / esz;
    const bool vec = aligned(a.logits, 16) && a.V % W == 0 && a.row_stride % W == 0 && a.req_stride % W == 0;
    if (dtype == CLK_DTYPE_BF16) {
        if (vec) return fused ? launch_verify<CLK_DTYPE_BF16, true, true>(a, L, s)
                              : launch_verify<CLK_DTYPE_BF16, true, false>(a, L, s);
        return fused ? launch_verify<CLK_DTYPE_BF16, false, true>(a, L, s)
                     : launch_verify<CLK_DTYPE_BF16, false, false>(a, L, s);
    }
    if (vec) return fused ? launch_verify<CLK_DTYPE_F32, true, true>(a, L, s)
                          : launch_verify<CLK_DTYPE_F32, true, false>(a, L, s);
    return fused ? launch_verify<CLK_DTYPE_F32, false, true>(a, L, s)
                 : launch_verify<CLK_DTYPE_F32, false, false>(a, L, s);
}

int verify_check(const void* d_logits, int32_t dtype, int64_t row_stride, int64_t req_stride, int32_t V, int32_t B,
                 const int32_t* d_block, const int32_t* d_len, int32_t* d_argmax, int32_t* d_accept,
                 int32_t* d_emitted, int32_t* d_out_tok)
{
    if (dtype != CLK_DTYPE_BF16 && dtype != CLK_DTYPE_F32) return CLK_EINVAL;
    if (V < 1 || B < 0 || B > CLK_MAX_BATCH) return CLK_EINVAL;
    if (row_stride < V || req_stride < 0) return CLK_EINVAL;
    if (B > 1 && req_stride < row_stride) return CLK_EINVAL;
    if (d_logits == nullptr || !aligned(d_logits, dtype == CLK_DTYPE_BF16 ? 2 : 4)) return CLK_EINVAL;
    if (!ok_i32(d_block) || !ok_i32(d_len) || !ok_i32(d_argmax) || !ok_i32(d_accept) || !ok_i32(d_emitted) ||
        !ok_i32(d_out_tok))
        return CLK_EINVAL;
    return CLK_OK;
}

}  // namespace clk

using namespace clk;

extern "C" int clk_verify_scratch_bytes(int32_t B, size_t* bytes)
{
    if (bytes == nullptr || B < 0 || B > CLK_MAX_BATCH) return CLK_EINVAL;
    *bytes = (size_t)(B > 0 ? B : 1) * (kBlock + 1) * sizeof(unsigned long long);
    return CLK_OK;
}

extern "C" int clk_verify_scratch_init(void* d_scratch, size_t bytes, clk_stream_t s)
{
    if (d_scratch == nullptr || !aligned(d_scratch, 8)) return CLK_EINVAL;
    return cuda_status(cudaMemsetAsync(d_scratch, 0, bytes, (cudaStream_t)s));
}

extern "C" int clk_verify_greedy(const void* d_logits, int32_t dtype, int64_t row_stride, int64_t req_stride,
                                 int32_t V, int32_t B, const int32_t* d_block, const int32_t* d_len,
                                 int32_t* d_argmax, int32_t* d_accept, int32_t* d_emitted, int32_t* d_out_tok,
                                 void* d_scratch, size_t scratch_bytes, clk_stream_t s)
{
    int rc = verify_check(d_logits, dtype, row_stride, req_stride, V, B, d_block, d_len, d_argmax, d_accept,
                          d_emitted, d_out_tok);
    if (rc != CLK_OK) return rc;
    if (B == 0) return CLK_OK;
    size_t need = 0;
    clk_verify_scratch_bytes(B, &need);
    if (d_scratch == nullptr || !aligned(d_scratch, 8) || scratch_bytes < need) return CLK_EINVAL;
    VerifyArgs a;
    a.logits = d_logits;
    a.row_stride = row_stride;
    a.req_stride = req_stride;
    a.V = V;
    a.B = B;
    a.block = d_block;
    a.len = d_len;
    a.len_hint = nullptr;
    a.argmax = d_argmax;
    a.accept = d_accept;
    a.emitted = d_emitted;
    a.out_tok = d_out_tok;
    a.keys = static_cast<unsigned long long*>(d_scratch);
    a.done = a.keys + (size_t)B * kBlock;
    a.slots = nullptr;
    a.late = 0;
    a.aligned = 0;
    LookupDev none = {};
    return verify_dispatch(a, dtype, false, none, (cudaStream_t)s);
}

extern "C" int clk_verify_append(clk_lookup* h, const int32_t* d_slots, const void* d_logits, int32_t dtype,
                                 int64_t row_stride, int64_t req_stride, int32_t V, int32_t B,
                                 const int32_t* d_block, const int32_t* d_len, const int32_t* d_len_hint,
                                 int32_t* d_argmax, int32_t* d_accept, int32_t* d_emitted, int32_t* d_out_tok,
                                 clk_stream_t s)
{
    int rc = check_batch(h, B);
    if (rc != CLK_OK) return rc;
    rc = verify_check(d_logits, dtype, row_stride, req_stride, V, B, d_block, d_len, d_argmax, d_accept, d_emitted,
                      d_out_tok);
    if (rc != CLK_OK) return rc;
    if (B == 0) return CLK_OK;
    if (!ok_i32(d_slots) || (d_len_hint != nullptr && !aligned(d_len_hint, 4))) return CLK_EINVAL;
    VerifyArgs a;
    a.logits = d_logits;
    a.row_stride = row_stride;
    a.req_stride = req_stride;
    a.V = V;
    a.B = B;
    a.block = d_block;
    a.len = d_len;
    a.len_hint = d_len_hint;
    a.argmax = d_argmax;
    a.accept = d_accept;
    a.emitted = d_emitted;
    a.out_tok = d_out_tok;
    const int par = h->vparity;
    a.keys = h->dev.vkeys + (size_t)par * (size_t)h->dev.max_slots * kBlock;
    a.done = h->dev.vdone + (size_t)par * (size_t)h->dev.max_slots;
    a.slots = d_slots;
    // It may overlap the proposal launch before it (unless the handle says
    // it is launched alone): the count of its CTAs that start behind that
    // launch is worked out at launch.
    a.late = h->alone ? 0 : 1;
    a.aligned = 0;
    rc = verify_dispatch(a, dtype, true, h->dev, (cudaStream_t)s);
    if (rc == CLK_OK) {
        h->vparity ^= 1;
        h->last_fused = kFusedGreedy;
        h->vsince = 1;
    } else {
        h->last_fused = kFusedNone;
    }
    return rc;
}

// ---------------------------------------------------------------------------
// Verification with library-owned scratch, for callers that cannot allocate.
// ---------------------------------------------------------------------------
// The scratch of clk_verify_greedy_static lives in this fixed device array
// instead of a caller buffer.  Every GPU that loads the library holds it
// until the process exits.  Device code could name it directly; host code
// must not pass its name to a kernel (on the host it is only a stand-in), so
// the entry point looks up its device address once per device.
static __device__ __align__(256) unsigned long long
    g_static_verify_scratch[(size_t)CLK_STATIC_VERIFY_MAX_BATCH * (kBlock + 1)];

#include <cuda.h>

#include <mutex>

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {nullptr};
unsigned long long g_static_ctx[kMaxDevices] = {0};  // id of the context the address belongs to

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Id of the calling thread's current context (0 on failure), through the
// driver entry points the runtime exposes (no link against the driver).
unsigned long long current_context_id()
{
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    if (get_current == nullptr || get_id == nullptr) {
        void* f1 = nullptr;
        void* f2 = nullptr;
        cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound, q2 = q1;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess)
            return 0;
        get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
        get_id = reinterpret_cast<CtxGetIdFn>(f2);
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the static scratch in the current context.  It is
// looked up on the first call on each device, and again whenever the
// device's current context is another one than at the last lookup (after
// cudaDeviceReset, say, the module is loaded anew, possibly elsewhere).
// nullptr on a CUDA error.
void* static_scratch_on_current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    const unsigned long long ctx = current_context_id();  // 0: none current yet on this thread
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (ctx == 0 || g_static_ptr[dev] == nullptr || g_static_ctx[dev] != ctx) {
        // (the lookup also makes the device's primary context current)
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_verify_scratch) != cudaSuccess || p == nullptr) return nullptr;
        const unsigned long long now = current_context_id();
        if (now == 0) return nullptr;
        g_static_ptr[dev] = p;
        g_static_ctx[dev] = now;
    }
    return g_static_ptr[dev];
}

}  // namespace

extern "C" int clk_verify_greedy_static(const void* d_logits, int32_t dtype, int64_t row_stride, int64_t req_stride,
                                        int32_t V, int32_t B, const int32_t* d_block, const int32_t* d_len,
                                        int32_t* d_argmax, int32_t* d_accept, int32_t* d_emitted,
                                        int32_t* d_out_tok, clk_stream_t s)
{
    if (B > CLK_STATIC_VERIFY_MAX_BATCH) return CLK_ECAPACITY;  // before the other checks: any larger B
    int rc = verify_check(d_logits, dtype, row_stride, req_stride, V, B, d_block, d_len, d_argmax, d_accept,
                          d_emitted, d_out_tok);
    if (rc != CLK_OK) return rc;
    if (B == 0) return CLK_OK;
    void* scratch = static_scratch_on_current_device();
    if (scratch == nullptr) return CLK_ECUDA;
    // The array keeps whatever the previous call left in it: clear the part
    // this call uses (the kernel needs its keys and counters at zero).
    const size_t used = (size_t)B * (kBlock + 1) * sizeof(unsigned long long);
    if (cudaMemsetAsync(scratch, 0, used, (cudaStream_t)s) != cudaSuccess) return CLK_ECUDA;
    VerifyArgs a;
    a.logits = d_logits;
    a.row_stride = row_stride;
    a.req_stride = req_stride;
    a.V = V;
    a.B = B;
    a.block = d_block;
    a.len = d_len;
    a.len_hint = nullptr;
    a.argmax = d_argmax;
    a.accept = d_accept;
    a.emitted = d_emitted;
    a.out_tok = d_out_tok;
    a.keys = static_cast<unsigned long long*>(scratch);
    a.done = a.keys + (size_t)B * kBlock;
    a.slots = nullptr;
    a.late = 0;
    a.aligned = 0;
    LookupDev none = {};
    return verify_dispatch(a, dtype, false, none, (cudaStream_t)s);
}

#ifdef CLK_TEST_HOOKS
// Test builds only (never in the shipped library): fill the static scratch
// with a byte, so that a test can show that clk_verify_greedy_static clears
// what it needs before it uses it.
extern "C" CLK_API int clk_test_fill_static_scratch(int byte, clk_stream_t s)
{
    void* scratch = static_scratch_on_current_device();
    if (scratch == nullptr) return CLK_ECUDA;
    return cuda_status(cudaMemsetAsync(scratch, byte, sizeof(g_static_verify_scratch), (cudaStream_t)s));
}
#endif
