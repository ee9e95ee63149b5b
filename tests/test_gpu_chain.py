"""The MLP chain with concurrent preprocessing (uw_mlp_forward, uw_mlp_autotune).

Each schedule -- everything fused, hard matrices preprocessed on a side
stream into one or two slots with or without an SM split, easy layers with a
palette-4 form made at load interleaved with hard ones, and the same plans run
serially -- must give, bit for bit, the output of the same layers computed
one call at a time by the uncompressed-weight kernels of the same variants
(uw_matmul_bf16) and uw_swiglu: the schedule changes only when the
preprocessing runs, never what a matmul computes.  A one-layer chain is also
checked against the fp64 oracle fed the GPU's own h.

Shapes: D = 512, F = 960 (30 row blocks of 32, an odd number of 64-column
groups in the down projection, a row count that is not a multiple of the
tensor-core tile), four layers with different sigmas; and two layers at the
measured model's shapes (4096 / 14336) at batch 256."""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu

D, F, LAYERS = 512, 960, 4


@pytest.fixture(scope="module")
def g(uw):
    from tests import _gpu
    return _gpu


def vid(uw, name):
    for v in range(uw.variant_count(uw.STRATEGY_FUSED)):
        if uw.variant_name(uw.STRATEGY_FUSED, v) == name:
            return v
    raise KeyError(name)


class Layer:
    def __init__(self, g, uw, ws_, seeds, sigma, d=D, f=F):
        self.mats = []
        for (rows, cols), seed in zip([(f, d), (f, d), (d, f)], seeds):
            w = wl.normal_weights(rows, cols, sigma, seed)
            c = g.Compressed(w)
            c.w_dev = g.dev_bits(w)
            c.p4 = torch.empty(uw.palette4_bytes(c.desc), dtype=torch.uint8, device="cuda")
            uw.transcode_palette4(c.desc, c.blob_dev, c.p4, ws_)
            self.mats.append(c)


def make_layers(g, uw, n, d=D, f=F, seed0=100):
    ws0 = g.workspace(1 << 16)
    layers = [Layer(g, uw, ws0, [seed0 + 3 * l + j for j in range(3)], 0.015 + 0.005 * l, d, f) for l in range(n)]
    torch.cuda.synchronize()
    assert uw.check_status(ws0) == 0
    return layers


@pytest.fixture(scope="module")
def layers(g, uw):
    return make_layers(g, uw, LAYERS)


def twin_chain(g, uw, layers, x_dev, variants):
    """The chain one call at a time on the original weights (variants[i]: matrix i)."""
    xin = x_dev
    batch = x_dev.shape[0]
    for l, L in enumerate(layers):
        outs = []
        for j, (c, xi) in enumerate(zip(L.mats[:2], (xin, xin))):
            y = g.empty_bits(batch, c.desc.rows)
            _twin(g, uw, c, xi, y, variants[3 * l + j])
            outs.append(y)
        h = g.empty_bits(batch, L.mats[0].desc.rows)
        uw.swiglu(outs[0], outs[1], h)
        y = g.empty_bits(batch, L.mats[2].desc.rows)
        _twin(g, uw, L.mats[2], h, y, variants[3 * l + 2])
        xin = y
    torch.cuda.synchronize()
    return g.host_bits(xin)


def _twin(g, uw, c, x, y, variant):
    ws = g.workspace(uw.workspace_size_bf16(c.desc.rows, c.desc.cols, x.shape[0], variant))
    uw.matmul_bf16(c.w_dev, x, y, ws, variant)


# variant of each strategy at each batch (the twin runs the same variant)
VARIANTS = {
    1: {"fused": "col_w16x1", "palette4": "col_w16x1", "exponent": "col_w16x1", "decompress": "col_w16x1"},
    4: {"fused": "w8s1", "palette4": "tc_g2", "exponent": "tc_g2", "decompress": "w8s1"},
    32: {"fused": "tc_g2", "palette4": "tc_g3", "exponent": "tc_g3", "decompress": "tc_g4"},
}
STRATEGY = {"fused": 1, "palette4": 2, "exponent": 3, "decompress": 0}

# (name, per-layer role strategies (with "easy" = palette-4 form made at load), slots, dec_ctas, side stream)
SCHEDULES = [
    ("fused_serial", lambda l: ["fused"] * 3, 2, 0, False),
    ("hard_double_split", lambda l: ["exponent", "palette4", "decompress"], 2, 16, True),
    ("hard_single", lambda l: ["exponent", "palette4", "decompress"], 1, 0, True),
    ("hard_serial", lambda l: ["exponent", "palette4", "decompress"], 2, 16, False),
    ("interleave_easy_hard", lambda l: ["easy"] * 3 if l % 2 == 0 else ["exponent", "decompress", "palette4"],
     2, 8, True),
    ("mixed_fused_hard", lambda l: ["fused", "exponent", "decompress"], 2, 40, True),
]


def build_chain(uw, layers, roles_of, batch):
    entries, variants = [], []
    for l, L in enumerate(layers):
        for c, role in zip(L.mats, roles_of(l)):
            strat = "palette4" if role == "easy" else role
            v = vid(uw, VARIANTS[batch][strat])
            entries.append((c.desc, c.blob_dev, c.p4 if role == "easy" else None,
                            uw.Plan(STRATEGY[strat], v, batch, 0.0)))
            variants.append(v)
    return entries, variants


@pytest.mark.parametrize("batch", [1, 4, 32])
@pytest.mark.parametrize("sched", SCHEDULES, ids=[s[0] for s in SCHEDULES])
def test_chain_equals_twin_layers(g, uw, layers, batch, sched):
    name, roles_of, slots, dec, use_side = sched
    entries, variants = build_chain(uw, layers, roles_of, batch)
    mats = uw.mlp_matrices(entries)
    x = g.dev_bits(wl.activations(batch, D, seed=batch))
    y = g.empty_bits(batch, D)
    s = uw.Schedule(slots, dec)
    ws = g.workspace(uw.mlp_workspace_size(mats, batch, s))
    side = torch.cuda.Stream() if use_side else None
    uw.mlp_forward(mats, x, y, ws, s, side_stream=side)
    assert uw.check_status(ws) == 0
    got = g.host_bits(y)
    ref = twin_chain(g, uw, layers, x, variants)
    assert np.array_equal(got, ref), "%s batch %d: %d of %d outputs differ" % (
        name, batch, int((got != ref).sum()), got.size)
    # a second call reuses the workspace (slots, split counters) and gives the same bits
    y2 = g.empty_bits(batch, D)
    uw.mlp_forward(mats, x, y2, ws, s, side_stream=side)
    assert uw.check_status(ws) == 0
    assert np.array_equal(g.host_bits(y2), ref)


def test_chain_back_to_back_calls(g, uw, layers):
    """Several forwards queued back to back on two streams, reading their
    inputs from the previous call's output, equal the same calls one at a time."""
    batch = 32
    entries, variants = build_chain(uw, layers, lambda l: ["exponent", "palette4", "decompress"], batch)
    mats = uw.mlp_matrices(entries)
    s = uw.Schedule(2, 24)
    ws = g.workspace(uw.mlp_workspace_size(mats, batch, s))
    side = torch.cuda.Stream()
    x = g.dev_bits(wl.activations(batch, D, seed=7))
    ys = [g.empty_bits(batch, D) for _ in range(4)]
    xin = x
    for y in ys:
        uw.mlp_forward(mats, xin, y, ws, s, side_stream=side)
        xin = y
    assert uw.check_status(ws) == 0
    ref_in = x
    for y in ys:
        ref = twin_chain(g, uw, layers, ref_in, variants)
        assert np.array_equal(g.host_bits(y), ref)
        ref_in = g.dev_bits(ref)


def test_chain_graph_capture(g, uw, layers):
    """The chain with a side stream captured into one CUDA graph and replayed."""
    batch = 32
    entries, variants = build_chain(uw, layers, lambda l: ["exponent", "palette4", "decompress"], batch)
    mats = uw.mlp_matrices(entries)
    s = uw.Schedule(2, 16)
    ws = g.workspace(uw.mlp_workspace_size(mats, batch, s))
    side = torch.cuda.Stream()
    x = g.dev_bits(wl.activations(batch, D, seed=11))
    y = g.empty_bits(batch, D)
    cap = torch.cuda.Stream()
    with torch.cuda.stream(cap):
        uw.mlp_forward(mats, x, y, ws, s, stream=cap, side_stream=side)  # warm-up: kernel attributes set
    cap.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        uw.mlp_forward(mats, x, y, ws, s, stream=cap, side_stream=side)
    y.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert uw.check_status(ws) == 0
    assert np.array_equal(g.host_bits(y), twin_chain(g, uw, layers, x, variants))


def test_one_layer_chain_against_oracle(g, uw, oracle, layers):
    batch = 4
    L = layers[1]
    entries, _ = build_chain(uw, [L], lambda l: ["exponent", "palette4", "decompress"], batch)
    mats = uw.mlp_matrices(entries)
    x = g.dev_bits(wl.activations(batch, D, seed=3))
    y = g.empty_bits(batch, D)
    s = uw.Schedule(2, 16)
    ws = g.workspace(uw.mlp_workspace_size(mats, batch, s))
    uw.mlp_forward(mats, x, y, ws, s, side_stream=torch.cuda.Stream())
    assert uw.check_status(ws) == 0
    # h as the chain computes it: the same variants one call at a time
    v = [e[3].variant for e in entries]
    gt, up, h = g.empty_bits(batch, F), g.empty_bits(batch, F), g.empty_bits(batch, F)
    _twin(g, uw, L.mats[0], x, gt, v[0])
    _twin(g, uw, L.mats[1], x, up, v[1])
    uw.swiglu(gt, up, h)
    torch.cuda.synchronize()
    y_ref, absum = oracle.matmul_f64(g.host_bits(h), L.mats[2].w)
    g.assert_within_bound(g.host_bits(y), y_ref, absum)


def test_chain_autotune(g, uw, layers):
    """The tuner returns plans and a split under which the concurrent chain
    equals the same plans run serially."""
    batch = 32
    entries, _ = build_chain(uw, layers, lambda l: ["easy"] * 3 if l == 0 else ["fused"] * 3, batch)
    mats = uw.mlp_matrices(entries)
    x = g.dev_bits(wl.activations(batch, D, seed=5))
    y = g.empty_bits(batch, D)
    ws = g.workspace(uw.mlp_autotune_workspace_size(mats, batch))
    side = torch.cuda.Stream()
    plans, sched = uw.mlp_autotune(mats, x, y, ws, passes=1, side_stream=side)
    assert len(plans) == 6 and all(p.us > 0 for p in plans)
    assert all(p.strategy == uw.STRATEGY_PALETTE4 for p in plans[3:])  # the matrices with a form
    assert sched.slots == 2 and sched.dec_ctas >= 0
    tuned = [(d, b, f, plans[i % 3 + (3 if f is not None else 0)]) for i, (d, b, f, p) in enumerate(entries)]
    tmats = uw.mlp_matrices(tuned)
    y1, y2 = g.empty_bits(batch, D), g.empty_bits(batch, D)
    uw.mlp_forward(tmats, x, y1, ws, sched, side_stream=side)
    uw.mlp_forward(tmats, x, y2, ws, sched, side_stream=None)
    assert uw.check_status(ws) == 0
    assert np.array_equal(g.host_bits(y1), g.host_bits(y2))


def test_chain_model_shapes_batch256(g, uw):
    """Two layers at the measured model's shapes, hard matrices on the side
    stream with an SM split, at batch 256."""
    batch = 256
    big = make_layers(g, uw, 2, d=wl.GATE_SHAPE[1], f=wl.GATE_SHAPE[0], seed0=500)
    roles = lambda l: ["exponent", "palette4", "decompress"] if l == 0 else ["palette4", "exponent", "fused"]
    entries, variants = [], []
    for l, L in enumerate(big):
        for c, role in zip(L.mats, roles(l)):
            v = vid(uw, "tc_g2")
            entries.append((c.desc, c.blob_dev, None, uw.Plan(STRATEGY[role], v, batch, 0.0)))
            variants.append(v)
    mats = uw.mlp_matrices(entries)
    x = g.dev_bits(wl.activations(batch, wl.GATE_SHAPE[1], seed=9))
    y = g.empty_bits(batch, wl.GATE_SHAPE[1])
    s = uw.Schedule(2, 32)
    ws = g.workspace(uw.mlp_workspace_size(mats, batch, s))
    uw.mlp_forward(mats, x, y, ws, s, side_stream=torch.cuda.Stream())
    assert uw.check_status(ws) == 0
    assert np.array_equal(g.host_bits(y), twin_chain(g, uw, big, x, variants))
