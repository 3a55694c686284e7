"""GPU parity of the tensor-core chunked kernel (tcgen05/TMEM/TMA) against the
fp64 oracle, through the C ABI: small cases spanning several chunks with ragged
tails, every n_h, gated/ungated, and the full-size workloads on sampled heads."""
import numpy as np
import pytest
import torch

import oracle
from deltaproduct_householder_product_gb300 import workloads as W
from tests.parity import assert_parity, err_stats

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dp():
    from deltaproduct_householder_product_gb300 import build
    build.build()
    import deltaproduct_householder_product_gb300 as dp
    assert torch.cuda.is_available()
    assert dp.supports("chunk_tc", 1, 64, 1, 128, 128, 2), "tensor-core kernel unavailable"
    return dp


def cuda(x):
    return {k: (None if v is None else v.cuda()) for k, v in x.items()}


def run(dp, x, impl="chunk_tc", h0=True, out_dtype=torch.float32, path="split"):
    """Forward through the C ABI; o in fp32 by default (the tolerance is on the
    kernel's arithmetic; a bf16 o adds its own final rounding, tested below).
    ``path`` "split" hands dp_forward the fast workspace (parallel prep kernel +
    state-pass kernel), "fused" only the minimum (one fused kernel)."""
    xc = cuda(x)
    size = workspace_for(dp, x, impl, path)
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    o, hf = dp.forward(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"],
                       xc["h0"] if h0 else None, impl=impl, workspace=ws, out_dtype=out_dtype)
    dp.check_status(ws)
    return o, hf


def workspace_for(dp, x, impl, path):
    """Workspace bytes selecting a path: "split" the fast size (one cooperative
    launch when the heads leave room, else prep + state-pass kernels),
    "split2" records only (always the two launches), "fused" the minimum."""
    if path == "split":
        return dp.workspace_size(*_dims(x), impl=impl, fast=True)
    lo = dp.workspace_size(*_dims(x), impl=impl)
    if path == "fused":
        return lo
    B, T, H, nh, _ = x["k"].shape
    ct = min(16, 32 // nh)
    return lo + ((B * H * (-(-T // ct)) * 18688 + 255) // 256) * 256


def _dims(x):
    B, T, H, nh, Dk = x["k"].shape
    return B, T, H, Dk, x["v"].shape[-1], nh, x["q"].dtype


def ref(x, h0=True):
    return oracle.forward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"] if h0 else None)


CASES = [(base, nh, T) for base in (W.BASE, W.NEARDUP, W.GATED, W.LONG)
         for nh, T in ((base.nh, 150),)] + [
    (W.BASE, 1, 200), (W.BASE, 3, 70), (W.BASE, 4, 33), (W.GATED, 1, 130), (W.GATED, 2, 97),
    (W.GATED, 3, 64), (W.NEARDUP, 2, 65), (W.LONG, 4, 1), (W.LONG, 1, 5), (W.GATED, 4, 17)]


@pytest.mark.parametrize("path", ["split", "fused"])
@pytest.mark.parametrize("base,nh,T", CASES, ids=lambda v: getattr(v, "name", str(v)))
def test_small_parity(dp, base, nh, T, path):
    w = base.scaled(B=2, H=3, T=T, nh=nh)
    x = W.make_inputs(w)
    o, hf = run(dp, x, path=path)
    ro, rh = ref(x)
    assert_parity(o, ro, "bf16", "o")
    assert_parity(hf, rh, "bf16", "h_final")


def test_repeated_launches_agree_bitwise(dp):
    """Every launch of the same inputs gives the same bits (the chunk paths
    use no atomics). The state pass's MMA groups hand TMEM results to one
    another (U' from the first group to the second, S to the next chunk); a
    hand-off not ordered through a commit shows up as a rare launch whose
    state diverges from one chunk on, about twice in a thousand fused
    launches of these cases when the second group was issued right behind
    the first. Small ungated and gated cases (n_h 2 and 3, ragged T),
    cooperative then fused, 2000 times over."""
    cases = [W.BASE.scaled(B=2, H=3, T=150, nh=2), W.NEARDUP.scaled(B=2, H=3, T=150, nh=3),
             W.GATED.scaled(B=2, H=3, T=150, nh=3)]
    xs = [cuda(W.make_inputs(w)) for w in cases]
    refs = [(run(dp, x, path="split"), run(dp, x, path="fused")) for x in xs]
    bad = []
    for rep in range(2000):
        for i, x in enumerate(xs):
            for j, path in enumerate(("split", "fused")):
                o, hf = run(dp, x, path=path)
                if not (torch.equal(o, refs[i][j][0]) and torch.equal(hf, refs[i][j][1])):
                    bad.append((rep, cases[i].name, path))
    assert not bad, f"{len(bad)} launches differ from the first, e.g. {bad[:5]}"


def test_workspace_sizes(dp):
    """The minimum workspace is the status block; the fast one adds one
    18688-byte record per (batch, head, chunk), chunks of min(16, 32 / n_h)
    tokens. The recurrent path needs no records."""
    for nh, T in ((1, 100), (2, 2048), (3, 31), (4, 8)):
        ct = min(16, 32 // nh)
        lo = dp.workspace_size(3, T, 5, 128, 128, nh, impl="chunk_tc")
        hi = dp.workspace_size(3, T, 5, 128, 128, nh, impl="chunk_tc", fast=True)
        assert lo == 256
        assert hi - lo >= 3 * 5 * (-(-T // ct)) * 18688 and (hi - lo) % 256 == 0
        assert dp.workspace_size(3, T, 5, 128, 128, nh, impl="recurrent", fast=True) == 256


@pytest.mark.parametrize("base,nh,T,h0", [(W.BASE, 2, 300, True), (W.GATED, 3, 77, True),
                                          (W.GATED, 1, 129, False), (W.NEARDUP, 4, 50, True),
                                          (W.LONG, 2, 17, False)],
                         ids=lambda v: getattr(v, "name", str(v)))
def test_split_modes_agree_bitwise(dp, base, nh, T, h0):
    """The cooperative launch and the two-kernel split mode share every
    arithmetic step (the same prep writes the same records, the same state
    pass reads them), so outputs and final states agree bit for bit. The
    fused mode solves the UT transform with another summation order: it
    meets the bf16 rule against the oracle, like the others."""
    x = W.make_inputs(base.scaled(B=2, H=3, T=T, nh=nh))
    o_s, h_s = run(dp, x, h0=h0, path="split")
    o_2, h_2 = run(dp, x, h0=h0, path="split2")
    assert torch.equal(o_s, o_2)
    assert torch.equal(h_s, h_2)
    o_f, h_f = run(dp, x, h0=h0, path="fused")
    ro, rh = ref(x, h0=h0)
    for o, h in ((o_s, h_s), (o_f, h_f)):
        assert_parity(o, ro, "bf16", "o")
        assert_parity(h, rh, "bf16", "h_final")


def test_forward_path_names_the_launch(dp):
    """dp_forward_path reports the mode each workspace size selects (a few
    heads leave room for the cooperative launch on a GB300)."""
    x = W.make_inputs(W.BASE.scaled(B=2, H=3, T=100))
    dims = (2, 100, 3, 128, 128, 2)
    for path, name in (("split", "chunk_coop"), ("split2", "chunk_split"), ("fused", "chunk_fused")):
        assert dp.forward_path(*dims, workspace_for(dp, x, "chunk_tc", path)) == name
    assert dp.forward_path(*dims, 256, impl="recurrent") == "recurrent"


def test_workspace_reuse_across_calls(dp):
    """The cooperative path keeps its record flags in the workspace; calls that
    reuse one workspace (different inputs, a shorter sequence, then the first
    inputs again) must each see only their own records."""
    xa = W.make_inputs(W.GATED.scaled(B=2, H=3, T=160, nh=2))
    xb = W.make_inputs(W.BASE.scaled(B=2, H=3, T=160, nh=2, seed=11))
    xc_ = W.make_inputs(W.BASE.scaled(B=2, H=3, T=70, nh=2, seed=12))
    ws = torch.zeros(workspace_for(dp, xa, "chunk_tc", "split"), dtype=torch.uint8, device="cuda")
    for x in (xa, xb, xc_, xa):
        g = cuda(x)
        o, hf = dp.forward(g["q"], g["k"], g["v"], g["beta"], g["g"], g["h0"], impl="chunk_tc",
                           workspace=ws, out_dtype=torch.float32)
        dp.check_status(ws)
        o_f, h_f = run(dp, x, path="split")   # the same mode on a fresh workspace
        assert torch.equal(o, o_f)
        assert torch.equal(hf, h_f)


def test_workspace_reuse_across_shapes(dp):
    """One workspace, zeroed once, reused by calls of different shapes: a
    split-mode problem with more than 4096 chunks (80 heads of the near-
    duplicate recipe) leaves record bytes all over the area where a small
    problem's cooperative flags live; the cooperative calls that follow
    (two seeds, another shape, the first seed again) must each equal the
    same call on a fresh zeroed workspace bit for bit and meet the bf16 rule
    against the oracle (DeltaProduct paper, Sec.4: the result depends on the
    inputs only, not on what earlier calls left in the scratch memory)."""
    big = W.NEARDUP.scaled(B=8, H=10, T=520)
    xb = cuda(W.make_inputs(big))
    size = workspace_for(dp, xb, "chunk_tc", "split")
    assert dp.forward_path(*_dims(xb)[:6], size) == "chunk_split"
    assert 8 * 10 * (-(-520 // 10)) > 4096
    small = [W.BASE.scaled(B=2, H=3, T=200, seed=21), W.BASE.scaled(B=2, H=3, T=200, seed=22),
             W.GATED.scaled(B=1, H=2, T=120, nh=3), W.BASE.scaled(B=2, H=3, T=200, seed=21)]
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    for w in small:
        assert size >= workspace_for(dp, W.make_inputs(w), "chunk_tc", "split")
    dp.forward(xb["q"], xb["k"], xb["v"], xb["beta"], xb["g"], xb["h0"], impl="chunk_tc", workspace=ws,
               out_dtype=torch.float32)
    dp.check_status(ws)
    for w in small:
        x = W.make_inputs(w)
        g = cuda(x)
        assert dp.forward_path(*_dims(g)[:6], size) == "chunk_coop"
        o, hf = dp.forward(g["q"], g["k"], g["v"], g["beta"], g["g"], g["h0"], impl="chunk_tc",
                           workspace=ws, out_dtype=torch.float32)
        dp.check_status(ws)
        o_f, h_f = run(dp, x, path="split")
        assert torch.equal(o, o_f), w
        assert torch.equal(hf, h_f), w
        ro, rh = ref(x)
        assert_parity(o, ro, "bf16", "o")
        assert_parity(hf, rh, "bf16", "h_final")


def test_coop_wait_timeout_is_reported(dp):
    """A device-side bounded wait that expires (failure detection, made to
    happen on purpose without a fault): the prep CTAs withhold the first
    record, so the state pass's wait for its flag runs out after a short
    limit. The call returns, the status word reads DP_ERR_TIMEOUT, the other
    heads' results are still right, and the next normal call on the same
    stream and workspace is clean and matches the oracle."""
    import time
    w = W.BASE.scaled(B=1, H=3, T=40)
    x = W.make_inputs(w)
    g = cuda(x)
    size = workspace_for(dp, x, "chunk_tc", "split")
    assert dp.forward_path(*_dims(g)[:6], size) == "chunk_coop"
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    ro, rh = ref(x)
    o = torch.zeros(w.B, w.T, w.H, w.Dv, dtype=torch.float32, device="cuda")
    try:
        dp.set_wait_fault(True, 4096)
        t0 = time.perf_counter()
        dp.forward(g["q"], g["k"], g["v"], g["beta"], g["g"], g["h0"], impl="chunk_tc", workspace=ws, out=o)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        dp.set_wait_fault()
    with pytest.raises(dp.DPError) as err:
        dp.check_status(ws)
    assert err.value.code == 6                        # DP_ERR_TIMEOUT
    assert elapsed < 10.0, elapsed                    # 4096 polls: milliseconds
    assert_parity(o[:, :, 1:], ro[:, :, 1:], "bf16", "o of the heads that were not starved")
    dp.check_status(ws)                               # read-and-clear: clean again
    o2, h2 = dp.forward(g["q"], g["k"], g["v"], g["beta"], g["g"], g["h0"], impl="chunk_tc", workspace=ws,
                        out_dtype=torch.float32)
    dp.check_status(ws)
    assert_parity(o2, ro, "bf16", "o after the timeout")
    assert_parity(h2, rh, "bf16", "h_final after the timeout")


def test_coop_pacing_wait_timeout_is_reported(dp):
    """The prep's pacing wait (it loads chunk c of a head only once the
    head's state pass has taken chunk c - 16) is bounded too: with the first
    record withheld, head 0's state pass never takes a chunk, so the prep's
    wait for its chunk 16 runs out as well (prep work queued behind it times
    out in turn). The call returns within the polls' time, reports
    DP_ERR_TIMEOUT, and the next normal call on the same workspace is clean
    and matches the oracle."""
    import time
    w = W.BASE.scaled(B=1, H=3, T=480)                 # 30 chunks per head (16 tokens each)
    x = W.make_inputs(w)
    g = cuda(x)
    size = workspace_for(dp, x, "chunk_tc", "split")
    assert dp.forward_path(*_dims(g)[:6], size) == "chunk_coop"
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    ro, rh = ref(x)
    o = torch.zeros(w.B, w.T, w.H, w.Dv, dtype=torch.float32, device="cuda")
    try:
        dp.set_wait_fault(True, 4096)
        t0 = time.perf_counter()
        dp.forward(g["q"], g["k"], g["v"], g["beta"], g["g"], g["h0"], impl="chunk_tc", workspace=ws, out=o)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        dp.set_wait_fault()
    with pytest.raises(dp.DPError) as err:
        dp.check_status(ws)
    assert err.value.code == 6                        # DP_ERR_TIMEOUT
    assert elapsed < 10.0, elapsed
    dp.check_status(ws)
    o2, h2 = dp.forward(g["q"], g["k"], g["v"], g["beta"], g["g"], g["h0"], impl="chunk_tc", workspace=ws,
                        out_dtype=torch.float32)
    dp.check_status(ws)
    assert_parity(o2, ro, "bf16", "o after the timeout")
    assert_parity(h2, rh, "bf16", "h_final after the timeout")


@pytest.mark.parametrize("base", [W.BASE, W.GATED, W.NEARDUP], ids=lambda w: w.name)
def test_bf16_output_is_rounded_fp32_output(dp, base):
    """The bf16-output variant runs the same arithmetic and only rounds the final
    store: it must equal the fp32 output rounded to nearest-even bf16, bit for bit."""
    x = W.make_inputs(base.scaled(B=1, H=2, T=200))
    o32, h32 = run(dp, x, out_dtype=torch.float32)
    o16, h16 = run(dp, x, out_dtype=torch.bfloat16)
    assert o16.dtype == torch.bfloat16
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(h16, h32)


def test_zero_initial_state_and_no_final(dp):
    w = W.GATED.scaled(B=1, H=2, T=100)
    x = W.make_inputs(w)
    xc = cuda(x)
    o, hf = dp.forward(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], None, impl="chunk_tc",
                       h_final=False, out_dtype=torch.float32)
    assert hf is None
    ro, _ = ref(x, h0=False)
    assert_parity(o, ro, "bf16", "o")


def test_gate_reset_and_beta_zero(dp):
    """g = 0 (reset) inside chunks and beta = 0 rows (pure decay): special cases
    the gated chunk algebra must handle without NaN/Inf."""
    w = W.GATED.scaled(B=1, H=2, T=90, nh=2)
    x = W.make_inputs(w)
    x["g"][:, 10] = 0.0
    x["g"][:, 45] = 0.0
    x["beta"][:, 20:40] = 0.0
    o, hf = run(dp, x)
    ro, rh = ref(x)
    assert_parity(o, ro, "bf16", "o")
    assert_parity(hf, rh, "bf16", "h_final")


@pytest.mark.parametrize("path", ["split", "split2", "fused"])
@pytest.mark.parametrize("nh", [1, 2, 3, 4])
def test_gated_rescale_schedule(dp, nh, path):
    """Gated chunks keep the state divided by the running product of chunk
    decays and rescale it only when that product would fall below e^-27:
    with gates in [0.3, 0.7] (a rescale every few chunks), runs of gates of
    exactly 1 (no decay) and exact zeros (a reset, which always rescales),
    outputs and final states still meet the bf16 rule against the oracle
    (DeltaProduct paper, Sec.4: H <- g_t H once per token)."""
    w = W.GATED.scaled(B=2, H=3, T=203, nh=nh)
    x = W.make_inputs(w)
    gen = torch.Generator().manual_seed(40 + nh)
    g = 0.3 + 0.4 * torch.rand(x["g"].shape, generator=gen)
    g[:, 40:90] = 1.0
    g[:, 17] = 0.0
    g[:, 150:153] = 0.0
    x["g"] = g.to(torch.bfloat16)
    o, hf = run(dp, x, path=path)
    ro, rh = ref(x)
    assert_parity(o, ro, "bf16", "o")
    assert_parity(hf, rh, "bf16", "h_final")


def test_matches_recurrent_kernel(dp):
    w = W.NEARDUP.scaled(B=1, H=4, T=256)
    x = W.make_inputs(w)
    o1, h1 = run(dp, x, "chunk_tc")
    o2, h2 = run(dp, x, "recurrent")
    ro, rh = ref(x)
    s1, s2 = err_stats(o1, ro), err_stats(o2, ro)
    assert s1["rel_max"] <= 2e-2 and s2["rel_max"] <= 2e-2, (s1, s2)


def sample_heads(x, pairs):
    """Sub-problem with the chosen (b, h) sequences as a batch of single heads."""
    out = {}
    for k in ("q", "k", "v", "beta", "g"):
        out[k] = None if x[k] is None else torch.stack([x[k][b, :, h] for b, h in pairs]).unsqueeze(2)
    out["h0"] = None if x["h0"] is None else torch.stack([x["h0"][b, h] for b, h in pairs]).unsqueeze(1)
    return out


def gather_heads(t, pairs, time_axis=True):
    """GPU result rows for the sampled (b, h) pairs, shaped like the oracle's."""
    if time_axis:
        return torch.stack([t[b, :, h] for b, h in pairs]).unsqueeze(2)
    return torch.stack([t[b, h] for b, h in pairs]).unsqueeze(1)


@pytest.mark.parametrize("base", [W.BASE, W.NEARDUP, W.GATED, W.LONG], ids=lambda w: w.name)
def test_full_size_sampled_heads(dp, base):
    """The full workload in the launch configuration the bench times; the oracle
    checks a few whole (batch, head) sequences."""
    x = W.make_inputs(base)
    o, hf = run(dp, x)
    rng = np.random.default_rng(7)
    n = 2 if base.T > 10000 else 3
    pairs = [(int(rng.integers(base.B)), int(rng.integers(base.H))) for _ in range(n)]
    sub = sample_heads(x, pairs)
    ro, rh = ref(sub)
    assert_parity(gather_heads(o, pairs), ro, "bf16", "o")
    assert_parity(gather_heads(hf, pairs, False), rh, "bf16", "h_final")


def test_state_carry_on_chunk_boundaries_is_bit_exact(dp):
    """When every call length is a multiple of the chunk (32 tokens at n_h = 2),
    carrying the state across calls runs exactly the same arithmetic (in the
    two-kernel split mode for every call: the segmented mode, which a longer
    call would take, adds the rounding of its combine)."""
    w = W.BASE.scaled(B=2, H=4, T=1024)
    x = W.make_inputs(w)
    xc = cuda(x)
    ws = torch.zeros(workspace_for(dp, x, "chunk_tc", "split2"), dtype=torch.uint8, device="cuda")
    assert dp.forward_path(*_dims(xc)[:6], ws.numel()) == "chunk_split"
    o_one, h_one = dp.forward(xc["q"], xc["k"], xc["v"], xc["beta"], impl="chunk_tc", workspace=ws,
                              out_dtype=torch.float32)
    state = torch.zeros_like(h_one)
    outs = []
    for s in range(4):
        sl = slice(s * 256, (s + 1) * 256)
        o_s, _ = dp.forward(xc["q"][:, sl].contiguous(), xc["k"][:, sl].contiguous(),
                            xc["v"][:, sl].contiguous(), xc["beta"][:, sl].contiguous(), None,
                            state, impl="chunk_tc", h_final=state, workspace=ws, out_dtype=torch.float32)
        outs.append(o_s)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(outs, 1), o_one)
    assert torch.equal(state, h_one)


SEG_CASES = [(W.BASE, 2, 805, True), (W.BASE, 2, 1027, False), (W.GATED, 4, 530, True), (W.GATED, 3, 700, False),
             (W.NEARDUP, 3, 651, True), (W.LONG, 1, 1100, True), (W.GATED, 1, 1040, True)]


@pytest.mark.parametrize("base,nh,T,h0", SEG_CASES, ids=lambda v: getattr(v, "name", str(v)))
def test_segmented_mode_parity(dp, base, nh, T, h0):
    """Few heads, long sequences: each sequence is cut into segments that run
    at once (from a zero state and from the identity), then chained and
    corrected (DeltaProduct paper, Sec.2 Eq.(1): the recurrence is affine in
    the state, so a segment's end state is A_s S_start + B_s). Outputs and
    final states meet the bf16 rule against the oracle; ragged segment tails,
    gates, h0 and every n_h."""
    w = base.scaled(B=1, H=2, T=T, nh=nh)
    x = W.make_inputs(w)
    xc = cuda(x)
    size = workspace_for(dp, x, "chunk_tc", "split")
    assert dp.forward_path(*_dims(xc)[:6], size) == "chunk_seg"
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    o, hf = dp.forward(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], xc["h0"] if h0 else None,
                       impl="chunk_tc", workspace=ws, out_dtype=torch.float32)
    dp.check_status(ws)
    ro, rh = ref(x, h0=h0)
    assert_parity(o, ro, "bf16", "o")
    assert_parity(hf, rh, "bf16", "h_final")
    # bf16 output: the same fp32 values rounded once; no final state asked for
    o16, none = dp.forward(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], xc["h0"] if h0 else None,
                           impl="chunk_tc", workspace=ws, out_dtype=torch.bfloat16, h_final=False)
    dp.check_status(ws)
    assert none is None
    assert torch.equal(o16, o.to(torch.bfloat16))


def test_long_state_carry_and_decode(dp):
    """8 carried 4096-token calls vs one 32768-token call, then 4096 decode steps
    continuing from the final state; checked against the oracle on sampled heads."""
    w = W.LONG
    x = W.make_inputs(w)
    xc = cuda(x)
    o_one, h_one = dp.forward(xc["q"], xc["k"], xc["v"], xc["beta"], None, None, impl="chunk_tc",
                              out_dtype=torch.float32)
    seg = w.T // W.LONG_CALLS
    state = torch.zeros_like(h_one)
    outs = []
    for s in range(W.LONG_CALLS):
        sl = slice(s * seg, (s + 1) * seg)
        o_s, _ = dp.forward(xc["q"][:, sl].contiguous(), xc["k"][:, sl].contiguous(),
                            xc["v"][:, sl].contiguous(), xc["beta"][:, sl].contiguous(), None,
                            state, impl="chunk_tc", h_final=state, out_dtype=torch.float32)
        outs.append(o_s)
    o_car = torch.cat(outs, 1)
    torch.cuda.synchronize()
    # with n_h = 3 a chunk holds 21 tokens, so 4096-token calls cut the chunk
    # grid elsewhere than one 32768-token call: both must meet the tolerance
    # against the oracle; their mutual difference is rounding only
    hs = [3, 11]
    pairs = [(0, h) for h in hs]
    sub = sample_heads(x, pairs)
    ro, rh = ref(sub)                                   # [2, T, 1, Dv], [2, 1, Dk, Dv]
    assert_parity(gather_heads(o_one, pairs), ro, "bf16", "o (single call)")
    assert_parity(gather_heads(h_one, pairs, False), rh, "bf16", "h_final (single call)")
    assert_parity(gather_heads(o_car, pairs), ro, "bf16", "o (8 carried calls)")
    assert_parity(gather_heads(state, pairs, False), rh, "bf16", "h_final (8 carried calls)")
    mutual = err_stats(o_car, o_one)
    assert mutual["rel_max"] <= 2e-2, mutual

    steps = 4096
    d = W.make_decode_inputs(w, steps)
    dc = cuda(d)
    st = h_one.clone()
    o_dec = torch.empty(steps, w.B, w.H, w.Dv, dtype=torch.float32, device="cuda")
    for i in range(steps):
        dp.decode_step(dc["q"][i], dc["k"][i], dc["v"][i], dc["beta"][i], None, st, out=o_dec[i])
    torch.cuda.synchronize()
    # the oracle runs the same decode inputs as one sequence from its own final state
    seq = {k: torch.stack([d[k][:, 0, h] for h in hs]).unsqueeze(2) for k in ("q", "k", "v", "beta")}
    rdo, rdh = oracle.forward(seq["q"], seq["k"], seq["v"], seq["beta"], None, rh)
    assert_parity(torch.stack([o_dec[:, 0, h] for h in hs]).unsqueeze(2), rdo, "bf16", "decode o")
    assert_parity(gather_heads(st, pairs, False), rdh, "bf16", "decode state")


@pytest.mark.parametrize("impl", ["chunk_tc", "recurrent"])
def test_linearity_in_h0_and_v(dp, impl):
    """o and h_final are linear in (h0, v) for fixed keys, betas and gates
    (DeltaProduct paper, Sec.4: the update is affine in H with an additive
    term in v). Doubling both doubles every intermediate exactly, so the
    outputs double bit for bit; two problems whose v and h0 add up to the
    original's (disjoint supports, so the sum is exact) give outputs that
    add up to the original's up to rounding (the bf16 rule)."""
    w = W.GATED.scaled(B=1, H=2, T=70, nh=2)
    x = W.make_inputs(w)
    xc = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    run = lambda v, h0: dp.forward(xc["q"], xc["k"], v, xc["beta"], xc["g"], h0, impl=impl,
                                   out_dtype=torch.float32)
    o1, h1 = run(xc["v"], xc["h0"])
    o2, h2 = run(2 * xc["v"], 2 * xc["h0"])
    assert torch.equal(o2, 2 * o1) and torch.equal(h2, 2 * h1)
    # additivity: split v and h0 into two problems with disjoint supports, so
    # that the parts sum to the originals exactly
    gen = torch.Generator().manual_seed(17)
    mv = (torch.rand(xc["v"].shape, generator=gen) < 0.5).cuda()
    mh = (torch.rand(xc["h0"].shape, generator=gen) < 0.5).cuda()
    zv, zh = torch.zeros_like(xc["v"]), torch.zeros_like(xc["h0"])
    oa, ha = run(torch.where(mv, xc["v"], zv), torch.where(mh, xc["h0"], zh))
    ob, hb = run(torch.where(mv, zv, xc["v"]), torch.where(mh, zh, xc["h0"]))
    assert_parity(oa + ob, o1.cpu().double().numpy(), "bf16", "additivity of o")
    assert_parity(ha + hb, h1.cpu().double().numpy(), "bf16", "additivity of h_final")
