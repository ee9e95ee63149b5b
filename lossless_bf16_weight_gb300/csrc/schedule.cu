// MLP chain executor with concurrent preprocessing, and its tuner (the
// Unweight blog's paragraphs on running the Huffman decoder or palette
// transcoder beside the reconstructive matmul, on the SM split between them,
// on "hard" and "easy" layers with double-buffered preprocess slots, and on
// tuning gate, then up, then down).
//
// The GPU work is the library's own kernels; this file only orders them:
// matmuls, SwiGLU and the easy matrices on the caller's stream, the hard
// matrices' preprocessing on a side stream, joined by events (one "ready"
// and one "free" event per slot).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "desc_check.h"
#include "kernels.h"
#include "uw.h"

namespace uw {
namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// What one matrix of the chain runs.
struct Step {
    int strategy = 0, variant = 0;
    int src = kSrcHuffman;  // what the matmul reads
    int pre = -1;           // preprocessing: -1 none, else the strategy whose form goes into a slot
    size_t form_bytes = 0;  // bytes the preprocessing writes
};

struct Chain {
    int64_t D = 0, Fmax = 0;
    std::vector<Step> steps;
    size_t control = 256;  // the matmuls' status word, split counters and partials
    size_t slot = 0;       // largest form a hard matrix writes
    int nhard = 0;
};

// Workspace: [control | x ping | x pong | g | u | h | slot 0 | slot 1 ...].
struct ChainLayout {
    size_t xa, xb, g, u, h, slots, slot_stride, total;
};

ChainLayout chain_layout(const Chain &c, int64_t batch, int slots) {
    ChainLayout L;
    const size_t xbytes = align256(size_t(batch) * size_t(c.D) * 2);
    const size_t fbytes = align256(size_t(batch) * size_t(c.Fmax) * 2);
    L.xa = align256(c.control);
    L.xb = L.xa + xbytes;
    L.g = L.xb + xbytes;
    L.u = L.g + fbytes;
    L.h = L.u + fbytes;
    L.slots = L.h + fbytes;
    L.slot_stride = align256(c.slot);
    L.total = L.slots + size_t(slots) * L.slot_stride;
    return L;
}

bool valid_desc(const uw_mlp_matrix &m) {
    return m.desc && m.blob_dev && desc_ok(*m.desc);
}

// Resolve every matrix's plan and size the workspace.  role_plans, when
// given, overrides the matrices' own plans: entries 0..2 (gate, up, down)
// for the matrices without a form, 3..5 for those with one (whose strategy
// stays PALETTE4).
uw_status plan_chain(const uw_mlp_matrix *m, int32_t n_layers, int64_t batch, const uw_plan *role_plans, Chain &c) {
    if (!m || n_layers <= 0 || batch <= 0)
        return UW_ERR_INVALID_ARG;
    for (int32_t i = 0; i < 3 * n_layers; i++)
        if (!valid_desc(m[i]))
            return UW_ERR_INVALID_ARG;
    c = Chain{};
    c.D = m[0].desc->cols;
    for (int32_t l = 0; l < n_layers; l++) {
        const uw_desc &g = *m[3 * l].desc, &u = *m[3 * l + 1].desc, &d = *m[3 * l + 2].desc;
        if (g.cols != c.D || u.cols != c.D || d.rows != c.D || u.rows != g.rows || d.cols != g.rows ||
            c.D % kGroup || g.rows % kGroup)
            return UW_ERR_SHAPE;  // the chain keeps whole 64-column groups (no ragged rows)
        c.Fmax = std::max<int64_t>(c.Fmax, g.rows);
    }
    c.steps.resize(size_t(3) * n_layers);
    for (int32_t i = 0; i < 3 * n_layers; i++) {
        const uw_desc &d = *m[i].desc;
        uw_plan pl = m[i].plan;
        if (role_plans) {
            pl = role_plans[i % 3 + (m[i].form_dev ? 3 : 0)];
            if (m[i].form_dev)
                pl.strategy = UW_STRATEGY_PALETTE4;
        }
        Step &s = c.steps[size_t(i)];
        uw_status st = plan_resolve(&pl, d, batch, &s.strategy, &s.variant);
        if (st != UW_OK)
            return st;
        const size_t n = size_t(d.rows) * size_t(d.cols);
        switch (s.strategy) {
            case UW_STRATEGY_FUSED:
                s.src = kSrcHuffman;
                break;
            case UW_STRATEGY_PALETTE4:
                s.src = kSrcPalette4;
                if (!m[i].form_dev) {
                    s.pre = UW_STRATEGY_PALETTE4;
                    s.form_bytes = n / 2;
                } else if (reinterpret_cast<uintptr_t>(m[i].form_dev) & 15) {
                    return UW_ERR_INVALID_ARG;
                }
                break;
            case UW_STRATEGY_EXPONENT:
                s.src = kSrcExponent;
                s.pre = UW_STRATEGY_EXPONENT;
                s.form_bytes = n;
                break;
            default:  // decompress, then the uncompressed kernel
                s.src = kSrcBf16;
                s.pre = UW_STRATEGY_DECOMPRESS_GEMM;
                s.form_bytes = 2 * n;
                break;
        }
        if (s.pre >= 0) {
            c.nhard++;
            c.slot = std::max(c.slot, s.form_bytes);
        }
        c.control = std::max(c.control, run_layout(d.rows, d.cols, batch, s.variant).weights);
    }
    return UW_OK;
}

int sched_slots(const uw_schedule *s) { return s ? s->slots : 2; }

uw_status check_sched(const uw_schedule *s) {
    if (s && (s->slots < 1 || s->slots > 2 || s->dec_ctas < 0))
        return UW_ERR_INVALID_ARG;
    return UW_OK;
}

// Events of one forward call, destroyed when it returns (a pending event
// is released once it completes).
struct Events {
    std::vector<cudaEvent_t> ev;
    ~Events() {
        for (cudaEvent_t e : ev)
            cudaEventDestroy(e);
    }
    bool make(size_t n) {
        for (size_t i = 0; i < n; i++) {
            cudaEvent_t e;
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
                return false;
            ev.push_back(e);
        }
        return true;
    }
};

uw_status cuda_ok(cudaError_t e) { return e == cudaSuccess ? UW_OK : UW_ERR_CUDA; }

uw_status run_chain(const uw_mlp_matrix *m, int32_t n_layers, const uint16_t *x, int64_t batch, uint16_t *y,
                    const Chain &c, const uw_schedule &sch, uint8_t *ws, size_t ws_bytes, cudaStream_t st,
                    cudaStream_t side) {
    const ChainLayout L = chain_layout(c, batch, sch.slots);
    if (ws_bytes < L.total)
        return UW_ERR_BUFFER_TOO_SMALL;
    const bool conc = side != nullptr && side != st;
    const int S = conc ? sch.slots : 1;
    uint32_t *status = reinterpret_cast<uint32_t *>(ws);
    uint16_t *xa = reinterpret_cast<uint16_t *>(ws + L.xa), *xb = reinterpret_cast<uint16_t *>(ws + L.xb);
    uint16_t *gb = reinterpret_cast<uint16_t *>(ws + L.g), *ub = reinterpret_cast<uint16_t *>(ws + L.u);
    uint16_t *hb = reinterpret_cast<uint16_t *>(ws + L.h);

    // events: ready[k], free[k] for each slot k, then fork and join
    Events E;
    if (conc && !E.make(size_t(2 * S + 2)))
        return UW_ERR_CUDA;
    cudaEvent_t *ready = conc ? E.ev.data() : nullptr, *freed = conc ? E.ev.data() + S : nullptr;
    uw_status s = UW_OK;
    if (conc) {
        cudaEvent_t fork = E.ev[size_t(2 * S)];
        if ((s = cuda_ok(cudaEventRecord(fork, st))) != UW_OK || (s = cuda_ok(cudaStreamWaitEvent(side, fork, 0))) != UW_OK)
            return s;
    }

    std::vector<int> hard;  // step index of each hard matrix, in the order of use
    for (size_t i = 0; i < c.steps.size(); i++)
        if (c.steps[i].pre >= 0)
            hard.push_back(int(i));
    int issued = 0, consumed = 0;
    auto slot_of = [&](int h) { return ws + L.slots + size_t(h % S) * L.slot_stride; };
    // Preprocess hard matrix h into slot h % S, once the matmul that read
    // the slot before (hard matrix h - S) has completed.
    auto preprocess = [&](int h) -> uw_status {
        const int i = hard[size_t(h)];
        const int k = h % S;
        cudaStream_t ps = conc ? side : st;
        if (conc && h >= S) {
            const uw_status e = cuda_ok(cudaStreamWaitEvent(side, freed[k], 0));
            if (e != UW_OK)
                return e;
        }
        BlobView v;
        fill_blob_view(*m[i].desc, m[i].blob_dev, &v);
        const int cap = conc ? sch.dec_ctas : 0;
        const Step &stp = c.steps[size_t(i)];
        const uw_status e =
            stp.pre == UW_STRATEGY_DECOMPRESS_GEMM
                ? launch_decompress(v, reinterpret_cast<uint16_t *>(slot_of(h)), status, ps, cap)
                : launch_transcode(v, slot_of(h), stp.pre == UW_STRATEGY_PALETTE4, status, ps, cap);
        if (e != UW_OK)
            return e;
        return conc ? cuda_ok(cudaEventRecord(ready[k], side)) : UW_OK;
    };
    auto top_up = [&]() -> uw_status {
        while (issued < int(hard.size()) && issued < consumed + S) {
            const uw_status e = preprocess(issued);
            if (e != UW_OK)
                return e;
            issued++;
        }
        return UW_OK;
    };
    auto matmul = [&](int i, const uint16_t *in, uint16_t *out) -> uw_status {
        uw_status e = top_up();
        if (e != UW_OK)
            return e;
        const Step &stp = c.steps[size_t(i)];
        const uw_desc &d = *m[i].desc;
        const WsLayout wl = run_layout(d.rows, d.cols, batch, stp.variant);
        GemvParams p{};
        fill_blob_view(d, m[i].blob_dev, &p.v);
        p.x = in;
        p.y = out;
        p.status = reinterpret_cast<uint32_t *>(ws + wl.status);
        p.counters = reinterpret_cast<uint32_t *>(ws + wl.counters);
        p.partial = reinterpret_cast<float *>(ws + wl.partial);
        p.rows = d.rows;
        p.cols = d.cols;
        p.batch = batch;
        const int h = consumed;
        if (stp.pre >= 0) {
            if (conc && (e = cuda_ok(cudaStreamWaitEvent(st, ready[h % S], 0))) != UW_OK)
                return e;
            if (stp.src == kSrcBf16)
                p.w = reinterpret_cast<const uint16_t *>(slot_of(h));
            else
                p.p4 = slot_of(h);
        } else if (stp.src == kSrcPalette4) {
            p.p4 = static_cast<const uint8_t *>(m[i].form_dev);
        }
        // beside a capped preprocess kernel, the persistent tensor-core CTAs
        // leave it its SMs (the sums do not depend on the CTA count)
        const int mm_cap = conc && sch.dec_ctas > 0 && sch.dec_ctas < sm_count() ? sm_count() - sch.dec_ctas : 0;
        if ((e = run_matmul(p, stp.variant, stp.src, st, mm_cap)) != UW_OK)
            return e;
        if (stp.pre >= 0) {
            if (conc && (e = cuda_ok(cudaEventRecord(freed[h % S], st))) != UW_OK)
                return e;
            consumed++;
            return top_up();
        }
        return UW_OK;
    };

    const uint16_t *xin = x;
    for (int32_t l = 0; l < n_layers && s == UW_OK; l++) {
        const int64_t F = m[3 * l].desc->rows;
        uint16_t *xout = l == n_layers - 1 ? y : (l % 2 == 0 ? xa : xb);
        if ((s = matmul(3 * l, xin, gb)) != UW_OK || (s = matmul(3 * l + 1, xin, ub)) != UW_OK ||
            (s = launch_swiglu(gb, ub, hb, batch * F, st)) != UW_OK || (s = matmul(3 * l + 2, hb, xout)) != UW_OK)
            break;
        xin = xout;
    }
    if (conc) {  // the caller's stream ends waiting for the side stream
        cudaEvent_t join = E.ev[size_t(2 * S + 1)];
        const uw_status e1 = cuda_ok(cudaEventRecord(join, side));
        const uw_status e2 = e1 == UW_OK ? cuda_ok(cudaStreamWaitEvent(st, join, 0)) : e1;
        if (s == UW_OK)
            s = e2;
    }
    return s;
}

// Tensor-core variants with two or three producer groups, by name.
std::vector<int> tc_variants() {
    std::vector<int> out;
    const int n = uw_variant_count(UW_STRATEGY_FUSED);
    for (int v = 0; v < n; v++) {
        const char *name = uw_variant_name(UW_STRATEGY_FUSED, v);
        if (name && (std::strncmp(name, "tc_g2", 5) == 0 || std::strncmp(name, "tc_g3", 5) == 0))
            out.push_back(v);
    }
    return out;
}

// Candidates of one role: the strategies (only PALETTE4 for the matrices
// with a form) with their default variant, and from batch 16 the
// tensor-core variants.
std::vector<uw_plan> role_candidates(int64_t batch, bool with_form) {
    std::vector<uw_plan> c;
    std::vector<int> strategies = {UW_STRATEGY_PALETTE4};
    if (!with_form)
        strategies = {UW_STRATEGY_FUSED, UW_STRATEGY_EXPONENT, UW_STRATEGY_PALETTE4, UW_STRATEGY_DECOMPRESS_GEMM};
    for (int st : strategies)
        c.push_back(uw_plan{st, -1, batch, 0.f});
    if (batch >= 16)
        for (int v : tc_variants())
            for (int st : strategies)
                c.push_back(uw_plan{st, v, batch, 0.f});
    return c;
}

}  // namespace
}  // namespace uw

using namespace uw;

extern "C" uw_status uw_mlp_workspace_size(const uw_mlp_matrix *m, int32_t n_layers, int64_t batch,
                                           const uw_schedule *sched, size_t *bytes) {
    if (!bytes)
        return UW_ERR_INVALID_ARG;
    uw_status s = check_sched(sched);
    if (s != UW_OK)
        return s;
    Chain c;
    if ((s = plan_chain(m, n_layers, batch, nullptr, c)) != UW_OK)
        return s;
    *bytes = chain_layout(c, batch, sched_slots(sched)).total;
    return UW_OK;
}

extern "C" uw_status uw_mlp_forward(const uw_mlp_matrix *m, int32_t n_layers, const uint16_t *x, int64_t batch,
                                    uint16_t *y, const uw_schedule *sched, void *ws, size_t ws_bytes, void *stream,
                                    void *side_stream) {
    if (!x || !y || !ws || (reinterpret_cast<uintptr_t>(x) & 15))
        return UW_ERR_INVALID_ARG;
    uw_status s = check_sched(sched);
    if (s != UW_OK)
        return s;
    Chain c;
    if ((s = plan_chain(m, n_layers, batch, nullptr, c)) != UW_OK)
        return s;
    const uw_schedule sch = sched ? *sched : uw_schedule{2, 0};
    return run_chain(m, n_layers, x, batch, y, c, sch, static_cast<uint8_t *>(ws), ws_bytes,
                     static_cast<cudaStream_t>(stream), static_cast<cudaStream_t>(side_stream));
}

extern "C" uw_status uw_mlp_autotune_workspace_size(const uw_mlp_matrix *m, int32_t n_layers, int64_t batch,
                                                    size_t *bytes) {
    if (!bytes)
        return UW_ERR_INVALID_ARG;
    size_t most = 0;
    for (const uw_plan &cand : role_candidates(batch, false)) {
        const uw_plan roles[6] = {cand, cand, cand, cand, cand, cand};
        Chain c;
        const uw_status s = plan_chain(m, n_layers, batch, roles, c);
        if (s == UW_ERR_INVALID_ARG || s == UW_ERR_SHAPE)
            return s;
        if (s == UW_OK)
            most = std::max(most, chain_layout(c, batch, 2).total);
    }
    *bytes = most;
    return most ? UW_OK : UW_ERR_INVALID_ARG;
}

extern "C" uw_status uw_mlp_autotune(const uw_mlp_matrix *m, int32_t n_layers, const uint16_t *x, int64_t batch,
                                     uint16_t *y, int32_t passes, uw_plan *plans_out, uw_schedule *sched_out,
                                     void *ws, size_t ws_bytes, void *stream, void *side_stream) {
    if (!m || n_layers <= 0 || !x || !y || !ws || !plans_out || !sched_out || passes <= 0 ||
        (reinterpret_cast<uintptr_t>(x) & 15))
        return UW_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream), side = static_cast<cudaStream_t>(side_stream);
    bool has_form[2] = {false, false};  // some matrix without / with a form
    for (int32_t i = 0; i < 3 * n_layers; i++)
        has_form[m[i].form_dev ? 1 : 0] = true;
    const std::vector<uw_plan> cands[2] = {role_candidates(batch, false), role_candidates(batch, true)};
    std::vector<int> decs = {0};  // SM splits to try (only with a side stream)
    if (side && side != st)
        for (int d : {8, 16, 24, 32, 48, 64})
            if (d < sm_count())
                decs.push_back(d);
    cudaEvent_t t0, t1;
    if (cudaEventCreate(&t0) != cudaSuccess)
        return UW_ERR_CUDA;
    if (cudaEventCreate(&t1) != cudaSuccess) {
        cudaEventDestroy(t0);
        return UW_ERR_CUDA;
    }
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    uw_status err = UW_OK;
    // median of 3 timed forwards after one warm-up; +inf for a plan that cannot run
    auto measure = [&](const uw_plan roles[6], int dec) -> double {
        Chain c;
        if (plan_chain(m, n_layers, batch, roles, c) != UW_OK)
            return INFINITY;
        const uw_schedule sch{2, dec};
        if (chain_layout(c, batch, 2).total > ws_bytes)
            return INFINITY;
        double t[3];
        for (int r = -1; r < 3; r++) {
            if (cudaEventRecord(t0, st) != cudaSuccess) {
                err = UW_ERR_CUDA;
                return INFINITY;
            }
            const uw_status s = run_chain(m, n_layers, x, batch, y, c, sch, wsb, ws_bytes, st, side);
            if (s == UW_ERR_UNSUPPORTED)
                return INFINITY;
            if (s != UW_OK) {
                err = s;
                return INFINITY;
            }
            float ms = 0.f;
            if (cudaEventRecord(t1, st) != cudaSuccess || cudaEventSynchronize(t1) != cudaSuccess ||
                cudaEventElapsedTime(&ms, t0, t1) != cudaSuccess) {
                err = UW_ERR_CUDA;
                return INFINITY;
            }
            if (r >= 0)
                t[r] = 1000.0 * ms;
        }
        std::sort(t, t + 3);
        return t[1];
    };
    // start: every role on its first candidate (fused, or palette-4 from the form)
    uw_plan roles[6] = {cands[0][0], cands[0][0], cands[0][0], cands[1][0], cands[1][0], cands[1][0]};
    int dec = 0;
    double best = measure(roles, dec);
    for (int pass = 0; pass < passes && err == UW_OK; pass++) {
        bool changed = false;
        for (int r = 0; r < 6 && err == UW_OK; r++) {
            if (!has_form[r / 3])
                continue;
            for (const uw_plan &cand : cands[r / 3]) {
                if (err != UW_OK)
                    break;
                uw_plan trial[6];
                std::copy(roles, roles + 6, trial);
                trial[r] = cand;
                const double t = measure(trial, dec);
                if (t < best * 0.99) {
                    best = t;
                    roles[r] = cand;
                    changed = true;
                }
            }
        }
        for (int d : decs) {
            if (d == dec || err != UW_OK)
                continue;
            const double t = measure(roles, d);
            if (t < best * 0.99) {
                best = t;
                dec = d;
                changed = true;
            }
        }
        if (!changed)
            break;
    }
    cudaEventDestroy(t0);
    cudaEventDestroy(t1);
    if (err != UW_OK)
        return err;
    if (!std::isfinite(best))
        return UW_ERR_UNSUPPORTED;
    for (int r = 0; r < 6; r++) {
        plans_out[r] = roles[r];
        plans_out[r].batch = batch;
        plans_out[r].us = float(best);
    }
    *sched_out = uw_schedule{2, dec};
    if (side && side != st && cudaStreamSynchronize(side) != cudaSuccess)
        return UW_ERR_CUDA;
    return cudaStreamSynchronize(st) == cudaSuccess ? UW_OK : UW_ERR_CUDA;
}
