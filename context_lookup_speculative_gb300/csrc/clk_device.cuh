// Device-side building blocks of the context-lookup hot path (sm_103a).
//
// Workspace layout (one caller-owned device buffer, see clk_lookup_workspace_bytes):
//   status  int32[64]                   latched device error (word 0) and its slot (word 1)
//   state   SlotState[max_slots]        scheduler state, history length, the last 64 tokens, counters
//   vkeys   u64[2][max_slots * 16]      fused verify: per-row packed (value, index) maxima
//   vdone   u64[2][max_slots]           fused verify: vectors verified per request
//                                       (two halves: consecutive fused verifies alternate)
//   skeys   u64[max_slots]              full-scan lookup: best (length, position) per request
//   ins     int4[2][max_slots]          per batch position: insertions a proposal left (see below)
//   hist    int32[max_slots][hstride]   token histories
//   tab     u32[max_slots][nlev][tsize] k-gram index, one table per match length
//
// The k-gram index.  For every match length k in [min_k, max_k] a slot owns an
// open-addressing table (linear probing, load <= 1/2) that maps a k-gram to
// the END position q of its most recent occurrence.  An entry is one 32-bit
// word: the low pos_bits bits hold q + 1 (pos_bits = the bit width of the
// history capacity) and the high bits a fingerprint of the k-gram's hash; 0
// is empty.  A k-gram ending at q is inserted once position q + 1 exists, so
// a table never returns the current suffix itself and every hit q gives a
// candidate j = q + 1 <= n - 1 with j >= k.  The longest suffix match of the
// pages' Step 1 is then the largest k whose table holds the suffix's k-gram,
// and its most recent occurrence is that table's entry: no chain walk and no
// history rescan, whatever the history length or its periodicity.  A
// fingerprint only filters: every stored occurrence is compared token by
// token before it is used or updated, so equal fingerprints of different
// k-grams never change an answer.  Entries are only ever inserted (the
// history only grows), so concurrent inserts use a CAS to claim an empty
// slot and an atomicMax on the same word (same fingerprint, larger q) to
// keep the most recent occurrence.
//
// Deferred inserts.  A slot records nidx, a history length up to which its
// tables are complete: they hold every k-gram ending at q <= nidx - 2.  The
// fused verify only writes the emitted tokens (n grows, nidx does not); the
// end positions nidx-1 .. n-2 stay pending until they are indexed, and every
// proposal checks the pending positions directly against the suffix (they
// are the most recent candidates) and the tables for everything older, so
// the answer is the same as with a complete index.  The proposal launch
// indexes them in dedicated warps: after its wait, beside its lookup warps;
// or, for small batches, it leaves at most kDeferMax of them to the next
// proposal launch, whose dedicated warps index them before that launch's
// wait, while the verify in between finishes.  A launch never raises nidx
// over entries it inserted itself: its ins record says what it leaves
// complete, and the next launch (which starts reading only once this one
// has completed) trusts that and raises nidx (atomicMax: it only grows
// between initialisations).
//
// The last kRing tokens of every history are also kept in the slot's record
// (ring[p mod kRing] = h[p]), next to n and the scheduler state, so that the
// proposal reads the state and the suffix window in one round trip.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "clk.h"

namespace clk {

constexpr int kBlock = CLK_BLOCK;
constexpr int kMaxK = CLK_MAX_K;
constexpr int kRing = 64;  // tokens of the history tail kept in the slot record
constexpr int kShort = 0;
constexpr int kLong = 1;

struct __align__(16) SlotState {
    int32_t n;
    int32_t mode;
    int32_t streak;
    int32_t miss;
    int32_t has_prev;
    int32_t cur_len;
    int32_t nidx;  // tables hold every k-gram ending at q <= nidx - 2
    int32_t pad1;
    int32_t ring[kRing];  // ring[p % kRing] = h[p] for the last kRing positions p < n
    long long steps, hits, long_steps, drafted, accepted, emitted;
    long long accept_hist[2][16];
};

struct LookupDev {
    int32_t* status;
    SlotState* state;
    unsigned long long* vkeys;
    unsigned long long* vdone;
    unsigned long long* skeys;  // full-scan lookup: packed (length, end + 1) per batch position
    int4* ins;                  // per batch position: index insertions left by the proposal launch
    int32_t* hist;
    uint32_t* tab;
    int64_t hstride;  // int32 elements per history
    int64_t cap;      // max_hist
    uint64_t tsize;   // entries per table (power of two)
    uint32_t posmask; // low bits of an entry: end position + 1
    uint32_t fpmask;  // high bits of an entry: fingerprint
    int32_t nlev;     // max_k - min_k + 1
    int32_t max_slots;
    int32_t vocab;
    int32_t pad;
    clk_params p;
};

__device__ __forceinline__ void latch(int32_t* status, int32_t code, int32_t detail)
{
    if (atomicCAS(status, 0, code) == 0) atomicExch(status + 1, detail);
}

__device__ __forceinline__ int32_t* hist_of(const LookupDev& L, int32_t slot)
{
    return L.hist + (int64_t)slot * L.hstride;
}

__device__ __forceinline__ uint32_t* table_of(const LookupDev& L, int32_t slot, int32_t level)
{
    return L.tab + ((uint64_t)slot * (uint64_t)L.nlev + (uint64_t)level) * L.tsize;
}

__device__ __forceinline__ bool token_ok(const LookupDev& L, int32_t t)
{
    return t >= 0 && (L.vocab <= 0 || t < L.vocab);
}

__device__ __forceinline__ int32_t long_len(const clk_params& p) { return 1 + p.head + p.tail; }
__device__ __forceinline__ int32_t short_len(const clk_params& p) { return 1 + p.head; }

// ---------------------------------------------------------------------------
// k-gram hashing: tokens taken backwards from the end position, w[l] = h[q-l].
// Each step xors a token in, multiplies by an odd 64-bit constant and folds
// the high half down; the final step mixes in k.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t kg_step(uint64_t acc, int32_t tok)
{
    acc ^= (uint32_t)tok;
    acc *= 0xFF51AFD7ED558CCDull;
    acc ^= acc >> 32;
    return acc;
}

__device__ __forceinline__ uint64_t kg_final(uint64_t acc, int32_t k)
{
    acc ^= (uint64_t)(uint32_t)k << 56;
    acc *= 0xC4CEB9FE1A85EC53ull;
    acc ^= acc >> 29;
    return acc;
}

constexpr uint64_t kHashSeed = 0x243F6A8885A308D3ull;

// True if h[p - l] == w[l] for l < k (the stored occurrence is the k-gram w).
// Loads go through L2 (ld.cg): the fused append compares against tokens that
// the same kernel has just written.
__device__ __forceinline__ bool kgram_at(const int32_t* h, int32_t p, const int32_t* w, int32_t k)
{
    if (p - (k - 1) < 0) return false;
    bool same = true;
#pragma unroll
    for (int l = 0; l < kMaxK; ++l)
        if (l < k) same &= (__ldcg(h + p - l) == w[l]);
    return same;
}

// The entry of the k-gram with hash H ending at q.
__device__ __forceinline__ uint32_t kg_entry(const LookupDev& L, uint64_t H, int32_t q)
{
    return ((uint32_t)(H >> 32) & L.fpmask) | (uint32_t)(q + 1);
}

// Insert k-gram w (ending at q, hash H) into one table; keeps the largest q.
// `same(p)` tells whether the k-gram ending at p equals w.  Linear probing
// from H mod tsize.  Returns false only if the table is full (cannot happen
// at load <= 1/2).
template <typename Same>
__device__ __forceinline__ bool index_insert(const LookupDev& L, uint32_t* tab, uint64_t H, int32_t q, Same same)
{
    const uint32_t mask = (uint32_t)(L.tsize - 1);
    const uint32_t entry = kg_entry(L, H, q);
    const uint32_t fp = entry & L.fpmask;
    uint32_t s = (uint32_t)H & mask;
    for (uint32_t probe = 0; probe <= mask; ++probe, s = (s + 1) & mask) {
        uint32_t cur = __ldcg(tab + s);
        if (cur == 0u) {
            const uint32_t old = atomicCAS(tab + s, 0u, entry);
            if (old == 0u) return true;
            cur = old;
        }
        if ((cur & L.fpmask) == fp && same((int32_t)(cur & L.posmask) - 1)) {
            atomicMax(tab + s, entry);
            return true;
        }
    }
    return false;
}

// index_insert for the latency-bound proposal launch: the probe sequence is
// read 8 entries per round trip (8 independent 4-byte loads), then the
// entries are examined in order.  Same result as index_insert.
template <typename Same>
__device__ __forceinline__ bool index_insert8(const LookupDev& L, uint32_t* tab, uint64_t H, int32_t q, Same same)
{
    const uint32_t mask = (uint32_t)(L.tsize - 1);
    const uint32_t entry = kg_entry(L, H, q);
    const uint32_t fp = entry & L.fpmask;
    uint32_t s = (uint32_t)H & mask;
    uint32_t probed = 0;
    while (probed <= mask) {
        uint32_t e[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) e[i] = __ldcg(tab + ((s + (uint32_t)i) & mask));
        // the first entry that is empty or carries the fingerprint
        int i0 = 8;
#pragma unroll
        for (int i = 7; i >= 0; --i)
            if (e[i] == 0u || (e[i] & L.fpmask) == fp) i0 = i;
        if (i0 == 8) {
            s = (s + 8u) & mask;
            probed += 8;
            continue;
        }
        uint32_t cur = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i == i0) cur = e[i];
        const uint32_t at = (s + (uint32_t)i0) & mask;
        if (cur == 0u) {
            const uint32_t old = atomicCAS(tab + at, 0u, entry);
            if (old == 0u) return true;
            cur = old;
        }
        if ((cur & L.fpmask) == fp && same((int32_t)(cur & L.posmask) - 1)) {
            atomicMax(tab + at, entry);
            return true;
        }
        // a different k-gram (same fingerprint, or a slot taken meanwhile):
        // continue after it
        s = (at + 1u) & mask;
        probed += (uint32_t)i0 + 1u;
    }
    return false;
}

// ---------------------------------------------------------------------------
// Step 3 (long-block scheduler).  sched_apply takes the slot's state fields
// already loaded, stores the new state and counters, and returns the block
// length; sched_update loads them first.
// ---------------------------------------------------------------------------
struct SchedFields {
    int32_t mode, streak, miss, has_prev;
};

__device__ __forceinline__ int32_t sched_apply(const clk_params& p, SlotState* st, SchedFields f, int32_t k,
                                               int32_t prev_a, int32_t prev_len)
{
    const bool flag = k >= p.tail_k;
    const bool near_full = f.has_prev && prev_a >= prev_len - 1 - p.near_full_slack;
    int32_t mode = f.mode, streak = f.streak, miss = f.miss;
    if (mode == kShort) {
        streak = (flag && near_full) ? streak + 1 : 0;
        if (streak >= p.enter_streak) {
            mode = kLong;
            miss = 0;
        }
    } else {
        miss = flag ? 0 : miss + 1;
        if (miss > p.sticky) {
            mode = kShort;
            streak = 0;
        }
    }
    const int32_t len = mode == kLong ? long_len(p) : short_len(p);
    st->mode = mode;
    st->streak = streak;
    st->miss = miss;
    st->has_prev = 1;
    st->cur_len = len;
    // Only this thread touches the slot's counters in the launch: additions
    // whose result nothing waits for (no load of the old values).
    auto add = [](long long* c, long long v) {
        if (v != 0) atomicAdd(reinterpret_cast<unsigned long long*>(c), (unsigned long long)v);
    };
    add(&st->steps, 1);
    add(&st->hits, (k >= p.min_k) ? 1 : 0);
    add(&st->long_steps, (p.tail > 0 && len == long_len(p)) ? 1 : 0);  // no tail: no long block
    add(&st->drafted, p.head + ((len == long_len(p) && k >= p.tail_k) ? p.tail : 0));
    return len;
}

__device__ __forceinline__ SchedFields sched_load(const SlotState* st)
{
    return SchedFields{st->mode, st->streak, st->miss, st->has_prev};
}

__device__ __forceinline__ int32_t sched_update(const clk_params& p, SlotState* st, int32_t k, int32_t prev_a,
                                                int32_t prev_len)
{
    return sched_apply(p, st, sched_load(st), k, prev_a, prev_len);
}

// ---------------------------------------------------------------------------
// Step 2 (fusion): decisions and the value of one block slot.
// ---------------------------------------------------------------------------
// agree_mask: bit i set when lookup draft token i equals draft-model proposal i.
__device__ __forceinline__ bool fuse_take_head(const clk_params& p, int32_t k, uint32_t agree_mask)
{
    if (k >= p.head_replace_k) return true;
    if (k < p.head_agree_k) return false;
    const uint32_t need = p.head_agree_n >= 32 ? 0xFFFFFFFFu : ((1u << p.head_agree_n) - 1u);
    return (agree_mask & need) == need;
}

__device__ __forceinline__ bool fuse_fill_tail(const clk_params& p, int32_t k, int32_t len)
{
    return len == long_len(p) && k >= p.tail_k;
}

// Slot i of the block given the decisions; c_prev = draft[i-1], m_prev = head[i-1].
__device__ __forceinline__ int32_t fuse_slot(const clk_params& p, int32_t i, int32_t last, bool take_head,
                                             bool fill_tail, int32_t c_prev, int32_t m_prev)
{
    if (i == 0) return last;
    if (i <= p.head) return take_head ? c_prev : m_prev;
    if (i <= p.head + p.tail) return fill_tail ? c_prev : CLK_SENT;
    return CLK_SENT;
}

// ---------------------------------------------------------------------------
// Commit of `count` tokens (in shared memory) to one slot: validation, the
// history write, the new length and the step counters.  The k-grams that the
// tokens complete are left for the index (nidx stays).  All threads of the
// block call it with the same arguments; sm_flag is 3 ints of shared
// memory; returns true if the tokens were written (uniform across the block).
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool block_commit_tokens(const LookupDev& L, int32_t slot, const int32_t* sm_tok,
                                                    int32_t count, int32_t* sm_flag)
{
    const int tid = threadIdx.x;
    SlotState* st = L.state + slot;
    if (tid == 0) {
        int ok = 1;
        const int32_t n = st->n;
        const int32_t len = st->cur_len;  // loaded with n: one round trip
        if (count < 0 || count > kBlock) {
            latch(L.status, CLK_EINVAL, slot);
            ok = 0;
        } else if ((int64_t)n + count > L.cap) {
            latch(L.status, CLK_ECAPACITY, slot);
            ok = 0;
        } else {
            for (int i = 0; i < count; ++i)
                if (!token_ok(L, sm_tok[i])) {
                    latch(L.status, CLK_EINVAL, slot);
                    ok = 0;
                    break;
                }
        }
        sm_flag[0] = ok;
        sm_flag[1] = n;
        sm_flag[2] = len;
    }
    __syncthreads();
    const bool ok = sm_flag[0] != 0;
    if (ok) {
        const int32_t n_old = sm_flag[1];
        int32_t* h = hist_of(L, slot);
        if (tid < count) {
            h[n_old + tid] = sm_tok[tid];
            st->ring[(n_old + tid) & (kRing - 1)] = sm_tok[tid];
        }
        if (tid == 0) {
            st->n = n_old + count;
            const int32_t len = sm_flag[2];
            if (len != 0 && count > 0) {
                // No other CTA touches this slot in the launch: the additions
                // need no return value, so nothing waits for them.
                atomicAdd(reinterpret_cast<unsigned long long*>(&st->accepted), (unsigned long long)(count - 1));
                atomicAdd(reinterpret_cast<unsigned long long*>(&st->emitted), (unsigned long long)count);
                if (count - 1 < 16) {
                    const int cls = (L.p.tail > 0 && len == long_len(L.p)) ? 1 : 0;
                    atomicAdd(reinterpret_cast<unsigned long long*>(&st->accept_hist[cls][count - 1]), 1ull);
                }
            }
            st->cur_len = 0;
        }
    }
    __syncthreads();
    return ok;
}

// Index every k-gram (all levels) that ends at q in [q_lo, q_hi], reading the
// tokens from the history.  Work items (q, level) are spread over the
// `nthr` threads whose rank is `rank`.  WIDE: probe 8 entries a round trip.
template <bool WIDE = false>
__device__ __forceinline__ void index_range(const LookupDev& L, int32_t slot, int32_t q_lo, int32_t q_hi,
                                            int32_t rank, int32_t nthr)
{
    if (q_hi < q_lo) return;
    const clk_params& p = L.p;
    const int32_t* h = hist_of(L, slot);
    const int64_t tasks = (int64_t)(q_hi - q_lo + 1) * L.nlev;
    for (int64_t task = rank; task < tasks; task += nthr) {
        const int32_t q = q_lo + (int32_t)(task / L.nlev);
        const int32_t lvl = (int32_t)(task % L.nlev);
        const int32_t k = p.min_k + lvl;
        if (q < k - 1) continue;
        int32_t w[kMaxK];
        uint64_t acc = kHashSeed;
#pragma unroll
        for (int l = 0; l < kMaxK; ++l) {
            if (l < k) {
                w[l] = __ldcg(h + q - l);
                acc = kg_step(acc, w[l]);
            }
        }
        auto same = [&](int32_t pos) { return kgram_at(h, pos, w, k); };
        const bool ok = WIDE ? index_insert8(L, table_of(L, slot, lvl), kg_final(acc, k), q, same)
                             : index_insert(L, table_of(L, slot, lvl), kg_final(acc, k), q, same);
        if (!ok) latch(L.status, CLK_ECAPACITY, slot);
    }
}

// The record of a proposal launch for batch position b, in ins[tag & 1][b]
// (tag != 0 names the launch): {tag, slot, z, w}.  Every k-gram of the slot
// ending before z - 1 is in the tables once the launch has completed; those
// ending at [z - 1, w - 2] are left to the next launch.  The next proposal
// launch reads the record of that tag after its wait, or, when it follows a
// fused greedy verify (so the recording launch has completed already),
// before it, and then runs the insertions while the verify finishes.  A
// proposal leaves at most kDeferMax positions this way, so that after one
// commit of at most kBlock tokens the next proposal still finds at most
// kDeferMax + kBlock pending, within its direct check; a record nobody takes
// costs only time.
constexpr int32_t kDeferMax = kBlock;
}  // namespace clk
