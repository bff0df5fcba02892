// Parameters, workspace layout, handle lifetime, status and inspection.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <new>

#include "clk.h"
#include "clk_device.cuh"
#include "clk_host.h"

using namespace clk;

namespace {

struct Layout {
    size_t status, state, vkeys, vdone, skeys, ins, hist, tab, total;
    int64_t hstride;
    uint64_t tsize;
    int32_t nlev;
    uint32_t posmask, fpmask;
};

// Fingerprint bits kept in an index entry.  A build may lower the limit to
// make equal fingerprints of different k-grams frequent (a test of the
// branches that tell them apart); answers never depend on it.
#ifndef CLK_TEST_FP_BITS
#define CLK_TEST_FP_BITS 32
#endif

uint64_t next_pow2(uint64_t x)
{
    uint64_t p = 1;
    while (p < x) p <<= 1;
    return p;
}

int layout_of(const clk_params* p, int32_t max_slots, int64_t max_hist, Layout* out)
{
    if (p == nullptr || clk_params_check(p) != CLK_OK) return CLK_EINVAL;
    if (max_slots < 1 || max_slots > (1 << 20)) return CLK_EINVAL;
    if (max_hist < 1 || max_hist > ((int64_t)1 << 30)) return CLK_EINVAL;
    Layout L;
    L.nlev = p->max_k - p->min_k + 1;
    L.hstride = (int64_t)align_up((size_t)max_hist, 64);
    L.tsize = next_pow2((uint64_t)(2 * max_hist) > 64 ? (uint64_t)(2 * max_hist) : 64);
    // An entry holds q + 1 <= max_hist - 1 in its low bits and a fingerprint
    // in the rest (at least one bit: max_hist <= 2^30).
    int pos_bits = 1;
    while (pos_bits < 31 && ((int64_t)1 << pos_bits) <= max_hist) ++pos_bits;
    L.posmask = (uint32_t)((1ull << pos_bits) - 1);
    const int fp_bits = (32 - pos_bits) < CLK_TEST_FP_BITS ? (32 - pos_bits) : CLK_TEST_FP_BITS;
    L.fpmask = (uint32_t)(((1ull << fp_bits) - 1) << pos_bits);
    const size_t ns = (size_t)max_slots;
    size_t off = 0;
    L.status = off;
    off = align_up(off + 64 * sizeof(int32_t), kAlign);
    L.state = off;
    off = align_up(off + ns * sizeof(SlotState), kAlign);
    L.vkeys = off;  // two halves, see clk_lookup::vparity
    off = align_up(off + 2 * ns * kBlock * sizeof(unsigned long long), kAlign);
    L.vdone = off;
    off = align_up(off + 2 * ns * sizeof(unsigned long long), kAlign);
    L.skeys = off;
    off = align_up(off + ns * sizeof(unsigned long long), kAlign);
    L.ins = off;
    off = align_up(off + 2 * ns * sizeof(int4), kAlign);  // two halves by tag parity
    L.hist = off;
    off = align_up(off + ns * (size_t)L.hstride * sizeof(int32_t), kAlign);
    L.tab = off;
    off = align_up(off + ns * (size_t)L.nlev * (size_t)L.tsize * sizeof(uint32_t), kAlign);
    L.total = off;
    *out = L;
    return CLK_OK;
}

}  // namespace

extern "C" void clk_params_default(clk_params* p)
{
    if (p == nullptr) return;
    p->min_k = 4;
    p->max_k = 12;
    p->head = 7;
    p->tail = 8;
    p->head_replace_k = 8;
    p->head_agree_k = 6;
    p->head_agree_n = 2;
    p->tail_k = 4;
    p->enter_streak = 2;
    p->sticky = 3;
    p->near_full_slack = 1;
}

extern "C" int clk_params_check(const clk_params* p)
{
    if (p == nullptr) return CLK_EINVAL;
    if (p->min_k < 1 || p->max_k < p->min_k || p->max_k > CLK_MAX_K) return CLK_EINVAL;
    if (p->head < 0 || p->tail < 0 || 1 + p->head + p->tail > CLK_BLOCK) return CLK_EINVAL;
    if (p->head_agree_n < 0 || p->head_agree_n > p->head) return CLK_EINVAL;
    if (p->head_replace_k < 0 || p->head_agree_k < 0 || p->tail_k < 0) return CLK_EINVAL;
    if (p->enter_streak < 1 || p->sticky < 0 || p->near_full_slack < 0) return CLK_EINVAL;
    return CLK_OK;
}

extern "C" const char* clk_status_string(int code)
{
    switch (code) {
    case CLK_OK: return "ok";
    case CLK_EINVAL: return "invalid argument";
    case CLK_ECAPACITY: return "capacity exceeded";
    case CLK_ECUDA: return "CUDA error";
    case CLK_ENOTIMPL: return "not implemented";
    case CLK_ESTATE: return "bad state";
    default: return "unknown status";
    }
}

extern "C" int clk_lookup_workspace_bytes(const clk_params* p, int32_t max_slots, int64_t max_hist, size_t* bytes)
{
    if (bytes == nullptr) return CLK_EINVAL;
    Layout L;
    int rc = layout_of(p, max_slots, max_hist, &L);
    if (rc != CLK_OK) return rc;
    *bytes = L.total;
    return CLK_OK;
}

extern "C" int clk_lookup_create(clk_lookup** h, const clk_params* p, int32_t max_slots, int64_t max_hist,
                                 int32_t vocab, void* d_workspace, size_t bytes)
{
    if (h == nullptr) return CLK_EINVAL;
    *h = nullptr;
    Layout L;
    int rc = layout_of(p, max_slots, max_hist, &L);
    if (rc != CLK_OK) return rc;
    if (d_workspace == nullptr || !aligned(d_workspace, kAlign) || bytes < L.total) return CLK_EINVAL;
    clk_lookup* hh = new (std::nothrow) clk_lookup;
    if (hh == nullptr) return CLK_EINVAL;
    char* base = static_cast<char*>(d_workspace);
    LookupDev& D = hh->dev;
    D.status = reinterpret_cast<int32_t*>(base + L.status);
    D.state = reinterpret_cast<SlotState*>(base + L.state);
    D.vkeys = reinterpret_cast<unsigned long long*>(base + L.vkeys);
    D.vdone = reinterpret_cast<unsigned long long*>(base + L.vdone);
    D.skeys = reinterpret_cast<unsigned long long*>(base + L.skeys);
    D.ins = reinterpret_cast<int4*>(base + L.ins);
    D.hist = reinterpret_cast<int32_t*>(base + L.hist);
    D.tab = reinterpret_cast<uint32_t*>(base + L.tab);
    D.hstride = L.hstride;
    D.cap = max_hist;
    D.tsize = L.tsize;
    D.posmask = L.posmask;
    D.fpmask = L.fpmask;
    D.nlev = L.nlev;
    D.max_slots = max_slots;
    D.vocab = vocab;
    D.pad = 0;
    D.p = *p;
    hh->ws = d_workspace;
    hh->bytes = L.total;
    hh->device = 0;
    hh->vparity = 0;
    hh->sparity = 0;
    hh->last_fused = kFusedNone;
    hh->ptag = 0;
    hh->defer_tag = 0;
    hh->vsince = 0;
    hh->alone = 0;
    cudaGetDevice(&hh->device);
    *h = hh;
    return CLK_OK;
}

extern "C" int clk_lookup_set_alone(clk_lookup* h, int32_t alone)
{
    if (!handle_ok(h)) return CLK_ESTATE;
    h->alone = alone != 0 ? 1 : 0;
    return CLK_OK;
}

extern "C" int clk_lookup_reset(clk_lookup* h, clk_stream_t s)
{
    if (!handle_ok(h)) return CLK_ESTATE;
    h->defer_tag = 0;
    return cuda_status(cudaMemsetAsync(h->ws, 0, h->bytes, (cudaStream_t)s));
}

extern "C" int clk_status(clk_lookup* h, int32_t* dev_status, int32_t* detail, clk_stream_t s)
{
    if (!handle_ok(h) || dev_status == nullptr) return CLK_EINVAL;
    int32_t st[2] = {0, 0};
    cudaStream_t cs = (cudaStream_t)s;
    if (cudaMemcpyAsync(st, h->dev.status, sizeof st, cudaMemcpyDeviceToHost, cs) != cudaSuccess) return CLK_ECUDA;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return CLK_ECUDA;
    *dev_status = st[0];
    if (detail) *detail = st[1];
    return CLK_OK;
}

extern "C" int clk_status_clear(clk_lookup* h, clk_stream_t s)
{
    if (!handle_ok(h)) return CLK_ESTATE;
    return cuda_status(cudaMemsetAsync(h->dev.status, 0, 2 * sizeof(int32_t), (cudaStream_t)s));
}

static int read_state(clk_lookup* h, int32_t slot, SlotState* out, clk_stream_t s)
{
    cudaStream_t cs = (cudaStream_t)s;
    if (cudaMemcpyAsync(out, h->dev.state + slot, sizeof(SlotState), cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        return CLK_ECUDA;
    return cuda_status(cudaStreamSynchronize(cs));
}

static void add_counters(clk_counters* c, const SlotState& st)
{
    c->steps += st.steps;
    c->hits += st.hits;
    c->long_steps += st.long_steps;
    c->drafted += st.drafted;
    c->accepted += st.accepted;
    c->emitted += st.emitted;
    for (int i = 0; i < 2; ++i)
        for (int j = 0; j < 16; ++j) c->accept_hist[i][j] += st.accept_hist[i][j];
}

extern "C" int clk_read_counters(clk_lookup* h, int32_t slot, clk_counters* out, clk_stream_t s)
{
    if (!handle_ok(h) || out == nullptr || slot < -1 || slot >= h->dev.max_slots) return CLK_EINVAL;
    memset(out, 0, sizeof *out);
    if (slot >= 0) {
        SlotState st;
        int rc = read_state(h, slot, &st, s);
        if (rc != CLK_OK) return rc;
        add_counters(out, st);
        return CLK_OK;
    }
    const size_t n = (size_t)h->dev.max_slots;
    SlotState* all = static_cast<SlotState*>(malloc(n * sizeof(SlotState)));
    if (all == nullptr) return CLK_EINVAL;
    cudaStream_t cs = (cudaStream_t)s;
    int rc = CLK_OK;
    if (cudaMemcpyAsync(all, h->dev.state, n * sizeof(SlotState), cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
        cudaStreamSynchronize(cs) != cudaSuccess)
        rc = CLK_ECUDA;
    if (rc == CLK_OK)
        for (size_t i = 0; i < n; ++i) add_counters(out, all[i]);
    free(all);
    return rc;
}

extern "C" int clk_read_slot_info(clk_lookup* h, int32_t slot, clk_slot_info* out, clk_stream_t s)
{
    if (!handle_ok(h) || out == nullptr || slot < 0 || slot >= h->dev.max_slots) return CLK_EINVAL;
    SlotState st;
    int rc = read_state(h, slot, &st, s);
    if (rc != CLK_OK) return rc;
    out->n = st.n;
    out->mode = st.mode;
    out->streak = st.streak;
    out->miss = st.miss;
    out->has_prev = st.has_prev;
    out->cur_len = st.cur_len;
    out->n_indexed = st.nidx;
    return CLK_OK;
}

extern "C" int clk_lookup_restore_state(clk_lookup* h, int32_t slot, const clk_slot_info* info,
                                        const clk_counters* counters, clk_stream_t s)
{
    if (!handle_ok(h) || info == nullptr || counters == nullptr || slot < 0 || slot >= h->dev.max_slots)
        return CLK_EINVAL;
    if ((info->mode != kShort && info->mode != kLong) || info->streak < 0 || info->miss < 0 ||
        (info->has_prev != 0 && info->has_prev != 1) || info->cur_len < 0 || info->cur_len > kBlock)
        return CLK_EINVAL;
    SlotState st;
    int rc = read_state(h, slot, &st, s);
    if (rc != CLK_OK) return rc;
    if (st.n != info->n) return CLK_EINVAL;
    st.mode = info->mode;
    st.streak = info->streak;
    st.miss = info->miss;
    st.has_prev = info->has_prev;
    st.cur_len = info->cur_len;
    st.steps = counters->steps;
    st.hits = counters->hits;
    st.long_steps = counters->long_steps;
    st.drafted = counters->drafted;
    st.accepted = counters->accepted;
    st.emitted = counters->emitted;
    for (int i = 0; i < 2; ++i)
        for (int j = 0; j < 16; ++j) st.accept_hist[i][j] = counters->accept_hist[i][j];
    cudaStream_t cs = (cudaStream_t)s;
    if (cudaMemcpyAsync(h->dev.state + slot, &st, sizeof st, cudaMemcpyHostToDevice, cs) != cudaSuccess)
        return CLK_ECUDA;
    return cuda_status(cudaStreamSynchronize(cs));  // the host copy of st dies with this call
}

extern "C" int clk_lookup_read_history(clk_lookup* h, int32_t slot, int32_t* h_out, int64_t cap, int64_t* n_out,
                                       clk_stream_t s)
{
    if (!handle_ok(h) || n_out == nullptr || slot < 0 || slot >= h->dev.max_slots || cap < 0) return CLK_EINVAL;
    if (cap > 0 && h_out == nullptr) return CLK_EINVAL;
    SlotState st;
    int rc = read_state(h, slot, &st, s);
    if (rc != CLK_OK) return rc;
    *n_out = st.n;
    const int64_t m = st.n < cap ? st.n : cap;
    if (m <= 0) return CLK_OK;
    cudaStream_t cs = (cudaStream_t)s;
    if (cudaMemcpyAsync(h_out, h->dev.hist + (int64_t)slot * h->dev.hstride, (size_t)m * sizeof(int32_t),
                        cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        return CLK_ECUDA;
    return cuda_status(cudaStreamSynchronize(cs));
}

extern "C" void clk_lookup_destroy(clk_lookup* h) { delete h; }
