// Lookup side of the hot path: prompt ingestion with the index build,
// incremental append, the suffix-match proposal, the scheduler and fusion
// (HyperQwen context-lookup article, "lookup 草稿的原理：三步走", Steps 1-3).
#include <cuda_runtime.h>
#include <stdint.h>

#include "clk.h"
#include "clk_device.cuh"
#include "clk_host.h"

namespace clk {

constexpr int kThreads = 256;

// Slot and prompt length of batch position b, validated; -1 slot if invalid.
__device__ __forceinline__ int32_t init_slot(const LookupDev& L, const int32_t* slots, const int64_t* off, int32_t b,
                                             int64_t* n_out)
{
    const int32_t slot = slots[b];
    if (slot < 0 || slot >= L.max_slots) return -1;
    const int64_t n = off[b + 1] - off[b];
    *n_out = n;
    return slot;
}

__global__ void k_init_state(LookupDev L, const int32_t* __restrict__ slots, const int64_t* __restrict__ off,
                             int32_t B)
{
    const int32_t b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int64_t n = 0;
    const int32_t slot = init_slot(L, slots, off, b, &n);
    if (slot < 0) {
        latch(L.status, CLK_EINVAL, b);
        return;
    }
    SlotState* st = L.state + slot;
    int32_t nn = (int32_t)n;
    if (n < 1) {
        latch(L.status, CLK_EINVAL, slot);
        nn = 0;
    } else if (n > L.cap) {
        latch(L.status, CLK_ECAPACITY, slot);
        nn = 0;
    }
    SlotState z = {};
    z.n = nn;
    z.nidx = nn;  // k_build_index indexes the whole prompt
    *st = z;
}

// Grid: B * chunks blocks; chunk c of batch position b copies positions
// [c*kThreads*4, (c+1)*kThreads*4).
__global__ void k_copy_prompt(LookupDev L, const int32_t* __restrict__ slots, const int32_t* __restrict__ prompt,
                              const int64_t* __restrict__ off, int32_t chunks)
{
    const int32_t b = blockIdx.x / chunks;
    const int64_t c = blockIdx.x % chunks;
    int64_t n = 0;
    const int32_t slot = init_slot(L, slots, off, b, &n);
    if (slot < 0 || n < 1 || n > L.cap) return;
    int32_t* h = hist_of(L, slot);
    int32_t* ring = L.state[slot].ring;
    const int32_t* src = prompt + off[b];
    bool bad = false;
    for (int64_t q = c * kThreads * 4 + threadIdx.x; q < min(n, (c + 1) * kThreads * 4); q += kThreads) {
        const int32_t t = src[q];
        bad |= !token_ok(L, t);
        h[q] = t;
        if (q >= n - kRing) ring[q  & (kRing - 1)] = t;
    }
    if (bad) latch(L.status, CLK_EINVAL, slot);
}

// Zero the tables of each slot in the batch.  Grid: B * chunks blocks.
__global__ void k_clear_tables(LookupDev L, const int32_t* __restrict__ slots, int32_t chunks, uint64_t per_chunk)
{
    const int32_t b = blockIdx.x / chunks;
    const uint64_t c = blockIdx.x % chunks;
    const int32_t slot = slots[b];
    if (slot < 0 || slot >= L.max_slots) return;
    const uint64_t total = (uint64_t)L.nlev * L.tsize;  // entries, a multiple of 4
    uint4* base = reinterpret_cast<uint4*>(table_of(L, slot, 0));
    const uint64_t lo = c * per_chunk, hi = min(total / 4, (c + 1) * per_chunk);
    for (uint64_t i = lo + threadIdx.x; i < hi; i += kThreads) base[i] = make_uint4(0u, 0u, 0u, 0u);
}

// Insert every eligible (end position, length) of each prompt: one thread per
// end position q <= n - 2, all lengths k <= q + 1.  Grid: B * chunks blocks.
__global__ void k_build_index(LookupDev L, const int32_t* __restrict__ slots, const int64_t* __restrict__ off,
                              int32_t chunks)
{
    const int32_t b = blockIdx.x / chunks;
    const int64_t c = blockIdx.x % chunks;
    int64_t n = 0;
    const int32_t slot = init_slot(L, slots, off, b, &n);
    if (slot < 0 || n < 1 || n > L.cap) return;
    const int64_t q = c * kThreads + threadIdx.x;
    if (q > n - 2) return;
    const int32_t* h = hist_of(L, slot);
    const clk_params& p = L.p;
    int32_t w[kMaxK];
#pragma unroll
    for (int l = 0; l < kMaxK; ++l) w[l] = (l < p.max_k && q - l >= 0) ? h[q - l] : CLK_SENT;
    uint64_t acc = kHashSeed;
#pragma unroll
    for (int l = 0; l < kMaxK; ++l) {
        const int32_t k = l + 1;
        if (k > p.max_k || q < k - 1) break;
        acc = kg_step(acc, w[l]);
        if (k >= p.min_k) {
            auto same = [&](int32_t pos) { return kgram_at(h, pos, w, k); };
            if (!index_insert(L, table_of(L, slot, k - p.min_k), kg_final(acc, k), (int32_t)q, same))
                latch(L.status, CLK_ECAPACITY, slot);
        }
    }
}

// One block per request: append d_tok[b][0..count) and index every k-gram
// not yet in the tables (the pending positions and the new ones).
__global__ void k_append(LookupDev L, const int32_t* __restrict__ slots, const int32_t* __restrict__ tok,
                         const int32_t* __restrict__ count)
{
    __shared__ int32_t sm_tok[kBlock];
    __shared__ int32_t sm_flag[3];
    __shared__ int32_t sm_nidx;
    const int32_t b = blockIdx.x;
    const int32_t slot = slots[b];
    if (slot < 0 || slot >= L.max_slots) {
        if (threadIdx.x == 0) latch(L.status, CLK_EINVAL, b);
        return;
    }
    const int32_t cnt = count[b];
    if (threadIdx.x < kBlock) sm_tok[threadIdx.x] = tok[(int64_t)b * kBlock + threadIdx.x];
    if (threadIdx.x == 0) sm_nidx = L.state[slot].nidx;
    __syncthreads();
    if (!block_commit_tokens(L, slot, sm_tok, cnt, sm_flag)) return;
    const int32_t n_new = sm_flag[1] + cnt;
    index_range(L, slot, max(sm_nidx - 1, 0), n_new - 2, threadIdx.x, blockDim.x);
    __syncthreads();
    if (threadIdx.x == 0) L.state[slot].nidx = n_new;
}

__device__ __forceinline__ bool warp_slot(const LookupDev& L, const int32_t* slots, int32_t B, int32_t* b_out,
                                          int32_t* slot_out)
{
    const int32_t b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (b >= B) return false;
    const int32_t slot = slots[b];
    *b_out = b;
    *slot_out = slot;
    return true;
}

// One thread per request.
__global__ void k_sched(LookupDev L, const int32_t* __restrict__ slots, int32_t B, const int32_t* __restrict__ k,
                        const int32_t* prev_a, const int32_t* prev_len, int32_t* len)
{
    const int32_t b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int32_t slot = slots[b];
    if (slot < 0 || slot >= L.max_slots) {
        latch(L.status, CLK_EINVAL, b);
        len[b] = short_len(L.p);
        return;
    }
    const int32_t pa = prev_a[b], pl = prev_len[b];
    len[b] = sched_update(L.p, L.state + slot, k[b], pa, pl);
}

// Fusion of one request by one warp; lanes < kBlock write the block.  Lane i
// holds lookup draft token i (c_lane) and draft-model proposal i (m_lane).
__device__ __forceinline__ void warp_fuse(const clk_params& p, int32_t last, int32_t c_lane, int32_t k,
                                          int32_t m_lane, int32_t len, int32_t* block_row)
{
    const unsigned full = 0xFFFFFFFFu;
    const int lane = threadIdx.x & 31;
    const unsigned agree = __ballot_sync(full, lane < p.head && c_lane == m_lane);
    const bool take_head = fuse_take_head(p, k, agree);
    const bool fill_tail = fuse_fill_tail(p, k, len);
    // slot i takes draft/head token i-1
    const int32_t c_prev = __shfl_up_sync(full, c_lane, 1);
    const int32_t m_prev = __shfl_up_sync(full, m_lane, 1);
    if (lane < kBlock) block_row[lane] = fuse_slot(p, lane, last, take_head, fill_tail, c_prev, m_prev);
}

// Stateless fusion: one warp per request.
__global__ void k_fuse(clk_params p, int32_t B, const int32_t* __restrict__ last_tok,
                       const int32_t* __restrict__ draft, const int32_t* __restrict__ k,
                       const int32_t* __restrict__ head, const int32_t* __restrict__ len,
                       int32_t* __restrict__ block)
{
    const int32_t b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (b >= B) return;
    const int lane = threadIdx.x & 31;
    const int32_t c_lane = lane < kBlock ? draft[(int64_t)b * kBlock + lane] : CLK_SENT;
    const int32_t m_lane = lane < p.head ? head[(int64_t)b * p.head + lane] : CLK_SENT;
    warp_fuse(p, last_tok[b], c_lane, k[b], m_lane, len[b], block + (int64_t)b * kBlock);
}

// Scheduler then fusion: one warp per request.
__global__ void k_fuse_sched(LookupDev L, const int32_t* __restrict__ slots, int32_t B,
                             const int32_t* __restrict__ draft, const int32_t* __restrict__ k,
                             const int32_t* __restrict__ head, const int32_t* prev_a, const int32_t* prev_len,
                             int32_t* len, int32_t* __restrict__ block)
{
    int32_t b, slot;
    if (!warp_slot(L, slots, B, &b, &slot)) return;
    const int lane = threadIdx.x & 31;
    const bool ok = slot >= 0 && slot < L.max_slots;
    int32_t l = short_len(L.p);
    const int32_t kk = k[b];
    if (lane == 0) {
        if (ok)
            l = sched_update(L.p, L.state + slot, kk, prev_a[b], prev_len[b]);
        else
            latch(L.status, CLK_EINVAL, b);
        len[b] = l;
    }
    l = __shfl_sync(0xFFFFFFFFu, l, 0);
    int32_t last = CLK_SENT;
    if (ok) {
        const int32_t n = L.state[slot].n;
        last = n >= 1 ? hist_of(L, slot)[n - 1] : CLK_SENT;
    }
    const int32_t c_lane = lane < kBlock ? draft[(int64_t)b * kBlock + lane] : CLK_SENT;
    const int32_t m_lane = lane < L.p.head ? head[(int64_t)b * L.p.head + lane] : CLK_SENT;
    warp_fuse(L.p, last, c_lane, kk, m_lane, l, block + (int64_t)b * kBlock);
}

// ---------------------------------------------------------------------------
// Full-scan lookup (the pages' own design, Step 1 of "三步走": scan the
// request's whole history; most candidates fail on their first tokens, the
// rest are extended up to max_k).  For every end position q <= n - 2 the
// match length m(q) = the number of tokens h[q - l] == h[n - 1 - l], l = 0..,
// capped at max_k; the answer is the largest (m, q) with m >= min_k, and
// j = q + 1.  Grid: B x chunks CTAs; each merges its best packed
// (m << 32 | q + 1) into skeys[b] with one atomicMax; k_scan_finish builds the
// draft and clears skeys.
// ---------------------------------------------------------------------------
constexpr int kScanPerCta = 4096;

__global__ void k_scan_match(LookupDev L, const int32_t* __restrict__ slots, int32_t chunks, int32_t per_cta)
{
    __shared__ int32_t sm_suf[kMaxK];
    __shared__ unsigned long long sm_red[kThreads / 32];
    const int32_t b = blockIdx.x / chunks;
    const int32_t c = blockIdx.x % chunks;
    const int32_t slot = slots[b];
    if (slot < 0 || slot >= L.max_slots) return;
    const int32_t n = L.state[slot].n;
    const int64_t lo64 = (int64_t)c * per_cta;
    if (lo64 >= n - 1) return;
    const int32_t lo = (int32_t)lo64, hi = (int32_t)min((int64_t)n - 1, lo64 + per_cta);  // end positions [lo, hi)
    if (n < 2 || lo >= hi) return;
    const clk_params& p = L.p;
    const int32_t* h = hist_of(L, slot);
    if (threadIdx.x < p.max_k) sm_suf[threadIdx.x] = threadIdx.x < n ? h[n - 1 - threadIdx.x] : CLK_SENT;
    __syncthreads();
    unsigned long long best = 0ull;
    for (int32_t q = lo + (int32_t)threadIdx.x; q < hi; q += kThreads) {
        int32_t m = 0;
        while (m < p.max_k && q - m >= 0 && h[q - m] == sm_suf[m]) ++m;
        if (m >= p.min_k) {
            const unsigned long long key = ((unsigned long long)m << 32) | (uint32_t)(q + 1);
            best = key > best ? key : best;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long v = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        best = v > best ? v : best;
    }
    if ((threadIdx.x & 31) == 0) sm_red[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kThreads / 32; ++w) best = sm_red[w] > best ? sm_red[w] : best;
        if (best != 0ull) atomicMax(L.skeys + b, best);
    }
}

// One warp per request: (k, j) from the merged key, the LZ77 draft.
__global__ void k_scan_finish(LookupDev L, const int32_t* __restrict__ slots, int32_t B, int32_t* __restrict__ draft,
                              int32_t* __restrict__ k_out, int32_t* __restrict__ j_out)
{
    const int32_t b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (b >= B) return;
    const int lane = threadIdx.x & 31;
    const int32_t slot = slots[b];
    const bool valid = slot >= 0 && slot < L.max_slots;
    const int32_t n = valid ? L.state[slot].n : 0;
    if (lane == 0) {
        if (!valid) latch(L.status, CLK_EINVAL, b);
        else if (n < 1) latch(L.status, CLK_ESTATE, slot);
    }
    const unsigned long long key = L.skeys[b];
    __syncwarp();
    if (lane == 0) L.skeys[b] = 0ull;
    int32_t k = 0, j = -1, c = CLK_SENT;
    if (valid && n >= 1 && key != 0ull) {
        k = (int32_t)(key >> 32);
        j = (int32_t)(uint32_t)key;
        if (lane < kBlock) c = hist_of(L, slot)[j + lane % (n - j)];
    }
    if (lane < kBlock) draft[(int64_t)b * kBlock + lane] = c;
    if (lane == 0) {
        k_out[b] = k;
        j_out[b] = j;
    }
}

constexpr int kMaxPending = 32;  // pending end positions checked directly
constexpr int kInsertWarps = 5;  // warps that index the pending positions
constexpr int kStepWarps = kMaxK + kInsertWarps;
static_assert(kMaxPending + kMaxK <= kRing, "the ring must cover the pending window");
static_assert(kDeferMax + kBlock <= kMaxPending, "what a launch leaves plus one commit stays within the direct check");

__device__ __forceinline__ void named_barrier(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Step 1 (and with FUSE, Steps 3 and 2) for one request per CTA.
//   Every warp loads the slot, then the slot's record: n, nidx, the
//   scheduler state and the last kRing tokens (one round trip, no barrier).
//   warps 0..nlev-1: one match length k = min_k + warp each.  The pending end
//     positions (not yet in the tables) are checked against the suffix from
//     the ring, most recent first; if none matches, 32 consecutive entries of
//     the table of length k are read at once from the k-gram's probe start,
//     and each one whose fingerprint matches (before the first empty entry)
//     is checked token by token by one warp-wide load, which also fetches the
//     16 tokens that follow the occurrence.
//   the last kInsertWarps warps: index pending positions, either before the
//     wait (those the previous proposal launch left in an ins record, see
//     deferred inserts in clk_device.cuh) or after it, beside the lookup
//     warps; the proposal never waits for them.  They raise nidx to what the
//     previous launch left complete; what this one indexes is published the
//     same way by the next launch (or by clk_lookup_append).
//   warp 0 then takes the longest level that matched (ballot), builds the
//   LZ77 draft, and with FUSE runs the scheduler and the fusion rule.
// 64 registers a thread: a CTA of up to 32 * kStepWarps threads fits an SM
// beside the verify launch's CTAs.
template <bool FUSE>
__global__ void __maxnreg__(64) k_lookup_step(
    LookupDev L, const int32_t* __restrict__ slots, const int32_t* __restrict__ head, const int32_t* prev_a,
    const int32_t* prev_len, int32_t* __restrict__ draft, int32_t* __restrict__ k_out, int32_t* __restrict__ j_out,
    int32_t* len_out, int32_t* __restrict__ block, int32_t early, int32_t tag, int32_t take, int32_t pre,
    int32_t defer)
{
    __shared__ __align__(16) int32_t sm_win[kStepWarps][kRing];  // each warp's copy of the ring (16-byte stores)
    __shared__ int32_t sm_q[kMaxK];
    __shared__ int32_t sm_follow[kMaxK][kBlock];
    const unsigned full = 0xFFFFFFFFu;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t b = blockIdx.x;
    const clk_params& p = L.p;
    const int nlev = L.nlev;

    // Launched as a programmatic dependent of the previous step's verify
    // launch, which commits the tokens this launch reads: wait for it.  This
    // step's verify launch may start streaming its first rows before (early:
    // the previous launch was a fused verify that uses the other half of its
    // scratch and let this launch start only after its own wait) or only
    // after that wait.
    if (early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // take != 0: the ins records of the previous proposal launch (tag take)
    // are read after the wait (that launch has completed by then).  pre: it
    // has completed already (a fused greedy verify waited for it before
    // letting this launch start), so the insert warps run the insertions it
    // left for this batch position now, while that verify finishes.
    int4 prev = make_int4(0, 0, 0, 0);
    const int4* prev_at = L.ins + (size_t)(take & 1) * (size_t)L.max_slots + b;
    if (pre && warp >= nlev) {
        prev = __ldcg(prev_at);
        if (prev.x == take && prev.y >= 0 && prev.y < L.max_slots && prev.z < prev.w)
            index_range<true>(L, prev.y, max(prev.z - 1, 0), prev.w - 2, tid - nlev * 32,
                              (int32_t)blockDim.x - nlev * 32);
    }
    // The slot, read once more after the wait: this early copy only lets the
    // record load go out together with that read.
    const int32_t slot_guess = slots[b];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // One round trip: the slot (every warp), the record of the slot read
    // before the wait (up to the end of the ring, 18 x 16 B), and for warp 0
    // the inputs that do not depend on it.  A slot that changed meanwhile
    // costs a second round trip for its record.
    const int32_t slot = __ldcg(slots + b);
    if (take != 0) prev = __ldcg(prev_at);
    int4 rec = make_int4(0, 0, 0, 0);
    const bool guess_ok = slot_guess >= 0 && slot_guess < L.max_slots;
    if (guess_ok && lane < 2 + kRing / 4) rec = __ldcg(reinterpret_cast<const int4*>(L.state + slot_guess) + lane);
    int32_t m_lane = CLK_SENT, pa = 0, pl = 0;
    if (FUSE && warp == 0) {
        if (lane < p.head) m_lane = head[(int64_t)b * p.head + lane];
        pa = prev_a[b];
        pl = prev_len[b];
    }
    const bool valid = slot >= 0 && slot < L.max_slots;
    if (slot != slot_guess) {
        rec = make_int4(0, 0, 0, 0);
        if (valid && lane < 2 + kRing / 4) rec = __ldcg(reinterpret_cast<const int4*>(L.state + slot) + lane);
    }
    // Keep the compiler from sinking round trip 1's loads to their first use
    // after the lookup: their values are needed by then anyway.
    if (FUSE) asm volatile("" ::"r"(m_lane), "r"(pa), "r"(pl));
    const int32_t n = __shfl_sync(full, rec.x, 0);
    int32_t nidx = min(__shfl_sync(full, rec.z, 1), n);
    // The previous launch's record for this request: every k-gram ending
    // before prev.z - 1 is in the tables (that launch completed), whatever
    // nidx says; nidx itself is raised only by a later launch (below), never
    // by the launch that made the insertions, so a lookup never trusts
    // entries still in flight.
    const bool prev_ok = take != 0 && prev.x == take && prev.y >= 0 && prev.y < L.max_slots && prev.z <= prev.w;
    const bool mine = prev_ok && prev.y == slot;
    if (mine) nidx = max(nidx, min(prev.z, n));
    int32_t* win = sm_win[warp];
    if (lane >= 2 && lane < 2 + kRing / 4) reinterpret_cast<int4*>(win)[lane - 2] = rec;
    __syncwarp();
    // 1: a request with a history; 2: a valid slot with an empty history (no
    // proposal; the scheduler still steps); 0: a bad slot.
    const int32_t ok = valid ? (n >= 1 ? 1 : 2) : 0;
    if (tid == 0) {
        if (!valid) latch(L.status, CLK_EINVAL, b);
        else if (ok == 2) latch(L.status, CLK_ESTATE, slot);
    }
    const int32_t* h = ok == 1 ? hist_of(L, slot) : nullptr;
    if (ok == 1 && n - nidx > kMaxPending) {
        // Many commits without a lookup in between: index them all first.
        index_range(L, slot, max(nidx - 1, 0), n - 2, tid, blockDim.x);
        __syncthreads();
        // (every warp of this CTA has read the slot's record by now)
        if (tid == 0) atomicMax(&L.state[slot].nidx, n);
        nidx = n;
    }
    const int32_t pend_lo = max(nidx - 1, 0);  // first end position not in the tables
    // nidx once the insert warps are done with the positions taken before
    // the wait.
    const int32_t covered = min(n, pre && mine && prev.z < prev.w ? max(nidx, prev.w) : nidx);
    // defer: at most kDeferMax positions still pending after that are left
    // to the next proposal launch; more are indexed here, after the wait.
    // The record says what this launch leaves complete (z) and to what
    // length the next one is to index (w).
    const bool deferred = defer && ok == 1 && n - covered <= kDeferMax;
    if (tag != 0 && tid == 0)
        L.ins[(size_t)(tag & 1) * (size_t)L.max_slots + b] = make_int4(tag, slot, deferred ? covered : n, n);
    const int32_t wlo = max(0, n - kRing);     // the ring holds positions [wlo, n)
    // Token at position x < n: from the ring when it holds x, else from the history.
    auto tok_at = [&](int32_t x) { return x >= wlo ? win[x  & (kRing - 1)] : __ldcg(h + x); };

    if (warp < nlev) {
        const int32_t k = p.min_k + warp;
        int32_t q = -1, fol = CLK_SENT;
        if (ok == 1 && n >= k + 1) {
            const int32_t cand = n - 2 - lane;
            bool m = cand >= max(pend_lo, k - 1);
            for (int l = 0; m && l < k; ++l) m = win[(cand - l)  & (kRing - 1)] == win[(n - 1 - l)  & (kRing - 1)];
            const unsigned hits = __ballot_sync(full, m);
            if (hits) {
                q = n - 2 - (__ffs(hits) - 1);
            } else {
                uint64_t acc = kHashSeed;
                for (int l = 0; l < k; ++l) acc = kg_step(acc, win[(n - 1 - l)  & (kRing - 1)]);
                const uint64_t H = kg_final(acc, k);
                const uint32_t fp = kg_entry(L, H, 0) & L.fpmask;
                const uint32_t mask = (uint32_t)(L.tsize - 1);
                const uint32_t* tab = table_of(L, slot, warp);
                const int32_t sl = lane < k ? win[(n - 1 - lane)  & (kRing - 1)] : 0;
                const uint32_t s0 = (uint32_t)H & mask;
                bool done = false;
                for (uint32_t probed = 0; !done && probed <= mask; probed += 32) {
                    const uint32_t e = __ldcg(tab + ((s0 + probed + (uint32_t)lane) & mask));
                    const unsigned empty = __ballot_sync(full, e == 0u);
                    const int lim = empty ? __ffs(empty) - 1 : 32;
                    unsigned cands = __ballot_sync(full, lane < lim && (e & L.fpmask) == fp);
                    done = empty != 0u;
                    while (cands) {
                        const int c = __ffs(cands) - 1;
                        cands &= cands - 1;
                        const int32_t pp = (int32_t)(__shfl_sync(full, e, c) & L.posmask) - 1;
                        bool same = true;
                        if (lane < k) same = pp < n && pp - lane >= 0 && tok_at(pp - lane) == sl;
                        int32_t f = CLK_SENT;
                        if (lane >= 16 && pp + 1 + (lane - 16) < n) f = tok_at(pp + 1 + (lane - 16));
                        if (__all_sync(full, same)) {
                            q = pp;
                            fol = f;
                            done = true;
                            break;
                        }
                    }
                }
            }
        }
        if (lane == 0) sm_q[warp] = q;
        if (lane >= 16) sm_follow[warp][lane - 16] = fol;
        __syncwarp();
        named_barrier(1, nlev * 32);
    } else {
        const int32_t ins_lo = max(covered - 1, 0);
        const int32_t rank = tid - nlev * 32, nthr = (int32_t)blockDim.x - nlev * 32;
        if (ok == 1 && n - 2 >= ins_lo && !deferred) {
            // Index the pending end positions, tokens from the ring.
            const int32_t tasks = (n - 1 - ins_lo) * nlev;
            for (int32_t task = rank; task < tasks; task += nthr) {
                const int32_t q = ins_lo + task / nlev;
                const int32_t lvl = task % nlev;
                const int32_t k = p.min_k + lvl;
                if (q < k - 1) continue;
                int32_t w[kMaxK];
                uint64_t acc = kHashSeed;
#pragma unroll
                for (int l = 0; l < kMaxK; ++l) {
                    if (l < k) {
                        w[l] = win[(q - l)  & (kRing - 1)];
                        acc = kg_step(acc, w[l]);
                    }
                }
                // One branch per check: the stored occurrence's k tokens from
                // the ring when it holds them all, else k loads issued together.
                auto same = [&](int32_t pos) {
                    if (pos - (k - 1) < 0 || pos >= n) return false;
                    if (pos - (k - 1) >= wlo) {
                        bool eq = true;
#pragma unroll
                        for (int l = 0; l < kMaxK; ++l)
                            if (l < k) eq &= win[(pos - l) & (kRing - 1)] == w[l];
                        return eq;
                    }
                    return kgram_at(h, pos, w, k);
                };
                if (!index_insert8(L, table_of(L, slot, lvl), kg_final(acc, k), q, same))
                    latch(L.status, CLK_ECAPACITY, slot);
            }
        }
        // Raise nidx to what the previous launch left complete.
        if (rank == 0 && prev_ok) atomicMax(&L.state[prev.y].nidx, prev.z);
        return;
    }
    if (warp != 0) return;
    int32_t kbest = 0, j = -1, c = CLK_SENT;
    if (ok == 1) {
        const int32_t lv = lane < nlev ? sm_q[lane] : -1;
        const unsigned hit = __ballot_sync(full, lv >= 0);
        if (hit) {
            const int best = 31 - __clz((int)hit);
            const int32_t q = __shfl_sync(full, lv, best);
            kbest = p.min_k + best;
            j = q + 1;
            if (lane < kBlock) {
                const int32_t idx = lane % (n - j);  // LZ77 copy at distance n - j
                c = q >= pend_lo ? win[(j + idx)  & (kRing - 1)] : sm_follow[best][idx];
            }
        }
    }
    if (lane < kBlock) draft[(int64_t)b * kBlock + lane] = c;
    if (lane == 0) {
        k_out[b] = kbest;
        j_out[b] = j;
    }
    if (FUSE) {
        // scheduler state from the record: (n, mode, streak, miss) in lane 0,
        // (has_prev, ...) in lane 1
        const int32_t has_prev = __shfl_sync(full, rec.x, 1);
        int32_t l = short_len(p);
        if (lane == 0) {
            if (ok != 0) l = sched_apply(p, L.state + slot, SchedFields{rec.y, rec.z, rec.w, has_prev}, kbest, pa, pl);
            len_out[b] = l;
        }
        l = __shfl_sync(full, l, 0);
        const int32_t last = ok == 1 ? win[(n - 1)  & (kRing - 1)] : CLK_SENT;
        warp_fuse(p, last, c, kbest, m_lane, l, block + (int64_t)b * kBlock);
    }
}

// One CTA per request, launched as a programmatic dependent of the previous
// launch in the stream (see k_lookup_step).
// Every launch records, per batch position, what it leaves complete in the
// index (ins records; the next launch raises nidx to it).  Batches of at
// most kDeferBatch requests also leave few pending insertions to the next
// launch: there the proposal is on the step's critical path, and the next
// one runs them before its wait, beside the verify's commit.  Larger
// batches index them after the wait, where the proposal overlaps the
// verify's streaming anyway.
constexpr int32_t kDeferBatch = 32;

template <bool FUSE>
int launch_lookup_step(clk_lookup* h, const int32_t* slots, int32_t B, const int32_t* head, const int32_t* prev_a,
                       const int32_t* prev_len, int32_t* draft, int32_t* k, int32_t* j, int32_t* len, int32_t* block,
                       cudaStream_t s)
{
    const LookupDev& L = h->dev;
    const int32_t early = h->last_fused == kFusedGreedy || h->last_fused == kFusedSampledPaired ? 1 : 0;
    // Tags alternate in parity (the record half), wrapping from 2^30 to 1.
    const int32_t tag = h->ptag = h->ptag >= (1 << 30) || h->ptag < 1 ? 1 : h->ptag + 1;
    const int32_t take = h->defer_tag;
    const int32_t pre = take != 0 && early && h->vsince ? 1 : 0;
    const int32_t defer = B <= kDeferBatch ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B);
    cfg.blockDim = dim3(32u * (unsigned)(L.nlev + kInsertWarps));  // <= 32 * kStepWarps
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int rc = cuda_status(cudaLaunchKernelEx(&cfg, k_lookup_step<FUSE>, L, slots, head, prev_a, prev_len, draft,
                                                  k, j, len, block, early, tag, take, pre, defer));
    h->defer_tag = rc == CLK_OK ? tag : 0;
    h->vsince = 0;
    return rc;
}

int proposal_cta_regs(int nlev)
{
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, k_lookup_step<true>) != cudaSuccess) return -1;
    return cta_regs(fa.numRegs, 32 * (nlev + kInsertWarps));
}

}  // namespace clk

using namespace clk;

extern "C" int clk_lookup_init(clk_lookup* h, const int32_t* d_slots, int32_t B, const int32_t* d_prompt,
                               const int64_t* d_prompt_off, clk_stream_t s)
{
    int rc = check_batch(h, B);
    if (rc != CLK_OK) return rc;
    if (B == 0) return CLK_OK;
    if (!ok_i32(d_slots) || !ok_i32(d_prompt) || d_prompt_off == nullptr || !aligned(d_prompt_off, 8))
        return CLK_EINVAL;
    const LookupDev& L = h->dev;
    cudaStream_t st = (cudaStream_t)s;
    h->defer_tag = 0;
    k_init_state<<<(B + 127) / 128, 128, 0, st>>>(L, d_slots, d_prompt_off, B);
    if ((rc = launch_status()) != CLK_OK) return rc;
    const int64_t copy_chunks = (L.cap + kThreads * 4 - 1) / (kThreads * 4);
    k_copy_prompt<<<(unsigned)(B * copy_chunks), kThreads, 0, st>>>(L, d_slots, d_prompt, d_prompt_off,
                                                                     (int32_t)copy_chunks);
    if ((rc = launch_status()) != CLK_OK) return rc;
    const uint64_t vec_total = (uint64_t)L.nlev * L.tsize / 4;  // uint4 stores per slot
    const uint64_t per_chunk = kThreads * 16;
    const int64_t clear_chunks = (int64_t)((vec_total + per_chunk - 1) / per_chunk);
    k_clear_tables<<<(unsigned)(B * clear_chunks), kThreads, 0, st>>>(L, d_slots, (int32_t)clear_chunks, per_chunk);
    if ((rc = launch_status()) != CLK_OK) return rc;
    const int64_t build_chunks = (L.cap + kThreads - 1) / kThreads;
    k_build_index<<<(unsigned)(B * build_chunks), kThreads, 0, st>>>(L, d_slots, d_prompt_off,
                                                                     (int32_t)build_chunks);
    return launch_status();
}

extern "C" int clk_lookup_append(clk_lookup* h, const int32_t* d_slots, int32_t B, const int32_t* d_tok,
                                 const int32_t* d_count, clk_stream_t s)
{
    int rc = check_batch(h, B);
    if (rc != CLK_OK) return rc;
    if (B == 0) return CLK_OK;
    if (!ok_i32(d_slots) || !ok_i32(d_tok) || !ok_i32(d_count)) return CLK_EINVAL;
    h->defer_tag = 0;  // this launch indexes every pending position
    k_append<<<B, 192, 0, (cudaStream_t)s>>>(h->dev, d_slots, d_tok, d_count);
    return launch_status();
}

extern "C" int clk_lookup_propose(clk_lookup* h, const int32_t* d_slots, int32_t B, int32_t* d_draft, int32_t* d_k,
                                  int32_t* d_j, clk_stream_t s)
{
    int rc = check_batch(h, B);
    if (rc != CLK_OK) return rc;
    if (B == 0) return CLK_OK;
    if (!ok_i32(d_slots) || !ok_i32(d_draft) || !ok_i32(d_k) || !ok_i32(d_j)) return CLK_EINVAL;
    return launch_lookup_step<false>(h, d_slots, B, nullptr, nullptr, nullptr, d_draft, d_k, d_j, nullptr,
                                     nullptr, (cudaStream_t)s);
}

extern "C" int clk_sched_step(clk_lookup* h, const int32_t* d_slots, int32_t B, const int32_t* d_k,
                              const int32_t* d_prev_accept, const int32_t* d_prev_len, int32_t* d_len, clk_stream_t s)
{
    int rc = check_batch(h, B);
    if (rc != CLK_OK) return rc;
    if (B == 0) return CLK_OK;
    if (!ok_i32(d_slots) || !ok_i32(d_k) || !ok_i32(d_prev_accept) || !ok_i32(d_prev_len) || !ok_i32(d_len))
        return CLK_EINVAL;
    k_sched<<<(B + 127) / 128, 128, 0, (cudaStream_t)s>>>(h->dev, d_slots, B, d_k, d_prev_accept, d_prev_len, d_len);
    return launch_status();
}

extern "C" int clk_fuse(const clk_params* p, int32_t B, const int32_t* d_last_tok, const int32_t* d_draft,
                        const int32_t* d_k, const int32_t* d_head, const int32_t* d_len, int32_t* d_block,
                        clk_stream_t s)
{
    if (p == nullptr || clk_params_check(p) != CLK_OK) return CLK_EINVAL;
    if (B < 0 || B > CLK_MAX_BATCH) return CLK_EINVAL;
    if (B == 0) return CLK_OK;
    if (!ok_i32(d_last_tok) || !ok_i32(d_draft) || !ok_i32(d_k) || (p->head > 0 && !ok_i32(d_head)) ||
        !ok_i32(d_len) || !ok_i32(d_block))
        return CLK_EINVAL;
    k_fuse<<<(B + 3) / 4, 128, 0, (cudaStream_t)s>>>(*p, B, d_last_tok, d_draft, d_k, d_head, d_len, d_block);
    return launch_status();
}

extern "C" int clk_fuse_sched(clk_lookup* h, const int32_t* d_slots, int32_t B, const int32_t* d_draft,
                              const int32_t* d_k, const int32_t* d_head, const int32_t* d_prev_accept,
                              const int32_t* d_prev_len, int32_t* d_len, int32_t* d_block, clk_stream_t s)
{
    int rc = check_batch(h, B);
    if (rc != CLK_OK) return rc;
    if (B == 0) return CLK_OK;
    if (!ok_i32(d_slots) || !ok_i32(d_draft) || !ok_i32(d_k) || (h->dev.p.head > 0 && !ok_i32(d_head)) ||
        !ok_i32(d_prev_accept) || !ok_i32(d_prev_len) || !ok_i32(d_len) || !ok_i32(d_block))
        return CLK_EINVAL;
    k_fuse_sched<<<(B + 3) / 4, 128, 0, (cudaStream_t)s>>>(h->dev, d_slots, B, d_draft, d_k, d_head, d_prev_accept,
                                                          d_prev_len, d_len, d_block);
    return launch_status();
}

extern "C" int clk_propose_fuse_sched(clk_lookup* h, const int32_t* d_slots, int32_t B, const int32_t* d_head,
                                      const int32_t* d_prev_accept, const int32_t* d_prev_len, int32_t* d_draft,
                                      int32_t* d_k, int32_t* d_j, int32_t* d_len, int32_t* d_block, clk_stream_t s)
{
    int rc = check_batch(h, B);
    if (rc != CLK_OK) return rc;
    if (B == 0) return CLK_OK;
    if (!ok_i32(d_slots) || (h->dev.p.head > 0 && !ok_i32(d_head)) || !ok_i32(d_prev_accept) ||
        !ok_i32(d_prev_len) || !ok_i32(d_draft) || !ok_i32(d_k) || !ok_i32(d_j) || !ok_i32(d_len) ||
        !ok_i32(d_block))
        return CLK_EINVAL;
    return launch_lookup_step<true>(h, d_slots, B, d_head, d_prev_accept, d_prev_len, d_draft, d_k, d_j, d_len,
                                    d_block, (cudaStream_t)s);
}

extern "C" int clk_lookup_propose_scan(clk_lookup* h, const int32_t* d_slots, int32_t B, int32_t ctas_per_request,
                                       int32_t* d_draft, int32_t* d_k, int32_t* d_j, clk_stream_t s)
{
    int rc = check_batch(h, B);
    if (rc != CLK_OK) return rc;
    if (ctas_per_request < 0) return CLK_EINVAL;
    if (B == 0) return CLK_OK;
    if (!ok_i32(d_slots) || !ok_i32(d_draft) || !ok_i32(d_k) || !ok_i32(d_j)) return CLK_EINVAL;
    // Each request's end positions [0, cap) are cut into `chunks` ranges of
    // per_cta positions, one CTA each.
    const int64_t cap = h->dev.cap;
    int64_t chunks = ctas_per_request > 0 ? ctas_per_request : (cap + kScanPerCta - 1) / kScanPerCta;
    if (chunks > cap) chunks = cap;
    const int64_t per_cta = (cap + chunks - 1) / chunks;
    if ((int64_t)B * chunks > 0x7FFFFFFF || per_cta > 0x7FFFFFFF) return CLK_EINVAL;
    k_scan_match<<<(unsigned)(B * chunks), kThreads, 0, (cudaStream_t)s>>>(h->dev, d_slots, (int32_t)chunks,
                                                                          (int32_t)per_cta);
    if ((rc = launch_status()) != CLK_OK) return rc;
    k_scan_finish<<<(B + 3) / 4, 128, 0, (cudaStream_t)s>>>(h->dev, d_slots, B, d_draft, d_k, d_j);
    return launch_status();
}
