"""GPU parity of the backward pass (dp_backward) against the fp64 oracle
backward, through the C ABI.

Every gradient (dq, dk, dv, dbeta, dg, dh0) is compared element by element
with oracle.backward on the same inputs and cotangents: small cases that
span several checkpoint segments with a ragged tail, every n_h, gated and
ungated, fp32 and bf16 inputs, fp32 and bf16 d_o; the degenerate sizes
(T = 0, T = 1, one segment exactly); and, at the bench workload's full size,
sampled heads against the oracle run on those heads alone plus a
directional derivative of the whole loss by central differences of the
forward oracle.

Tolerance: the kernel runs in fp32 on inputs the oracle sees exactly (bf16
upcasts exactly), so errors come from fp32 rounding (unit 6e-8) of the
recurrence and of the gradient sums: about sqrt(T n_h D) accumulated
roundings for the longest dependency chain, 4e-5 relative at the bench
size (T n_h = 4096, D = 128). Each gradient tensor must satisfy
max|err| <= TOL_REL * RMS(reference) with TOL_REL = 1e-4 (observed: about
2e-6 on the small cases).
"""
import numpy as np
import pytest
import torch

import oracle
from deltaproduct_householder_product_gb300 import workloads as W
from tests.parity import err_stats

pytestmark = pytest.mark.gpu

TOL_REL = 1e-4
NAMES = ("dq", "dk", "dv", "dbeta", "dg", "dh0")


@pytest.fixture(scope="module")
def dp():
    from deltaproduct_householder_product_gb300 import build
    build.build()
    import deltaproduct_householder_product_gb300 as dp
    assert torch.cuda.is_available()
    return dp


def cotangents(w, seed, do_dtype=torch.float32):
    gen = torch.Generator().manual_seed(seed)
    d_o = torch.randn(w.B, w.T, w.H, w.Dv, generator=gen).to(do_dtype)
    dhf = torch.randn(w.B, w.H, w.Dk, w.Dv, generator=gen)
    return d_o, dhf


def run_both(dp, w, d_o, dhf, heads=None, impl="auto"):
    x = W.make_inputs(w)
    xc = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    got = dp.backward(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], xc["h0"], d_o=d_o.cuda(),
                      dh_final=None if dhf is None else dhf.cuda(), impl=impl)
    torch.cuda.synchronize()
    if heads is None:
        ref = oracle.backward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], d_o, dhf)
        return got, ref, None
    return got, x, heads


def check(got, ref, what, tol=TOL_REL):
    stats = {}
    for n in NAMES:
        if ref[n] is None:
            assert got[n] is None, n
            continue
        s = err_stats(got[n], ref[n])
        stats[n] = s
        assert s["rel_max"] <= tol, f"{what} {n}: {s}"
    return stats


CASES = [
    ("tiny-f32", W.TINY.scaled(T=29), 0),
    ("d64-f32-gated", W.TINY.scaled(Dk=64, Dv=64, T=53, nh=3, gated=True, h0_std=0.02), 1),
    ("base-nh1", W.BASE.scaled(B=2, H=2, T=40, nh=1), 2),
    ("base-nh2", W.BASE.scaled(B=2, H=2, T=37), 3),
    ("neardup-nh3", W.NEARDUP.scaled(B=1, H=2, T=30), 4),
    ("gated-nh4", W.GATED.scaled(B=2, H=1, T=27), 5),
    ("long-nh3-one-segment", W.LONG.scaled(B=1, H=3, T=12), 6),
]


@pytest.mark.parametrize("name,w,seed", CASES, ids=[c[0] for c in CASES])
def test_backward_parity(dp, name, w, seed):
    d_o, dhf = cotangents(w, 100 + seed)
    got, ref, _ = run_both(dp, w, d_o, dhf)
    stats = check(got, ref, name)
    print(name, {n: round(s["rel_max"], 8) for n, s in stats.items()})


def test_backward_bf16_cotangent_and_no_dh_final(dp):
    w = W.GATED.scaled(B=1, H=2, T=26, nh=2)
    d_o, _ = cotangents(w, 120, torch.bfloat16)
    got, ref, _ = run_both(dp, w, d_o, None)
    check(got, ref, "bf16 d_o")


@pytest.mark.parametrize("T", [0, 1])
def test_backward_degenerate_lengths(dp, T):
    w = W.GATED.scaled(B=2, H=2, T=T, nh=2)
    d_o, dhf = cotangents(w, 130 + T)
    got, ref, _ = run_both(dp, w, d_o, dhf)
    if T == 0:
        assert torch.equal(got["dh0"].cpu(), dhf)
    else:
        check(got, ref, f"T={T}")


def test_backward_full_size_sampled_heads(dp):
    """Bench workload (B4 H8 T2048 n_h 2): the first and last heads against
    the oracle run on those heads alone."""
    w = W.BASE
    d_o, dhf = cotangents(w, 140)
    got, x, _ = run_both(dp, w, d_o, dhf, heads=True)
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        sl = lambda t: None if t is None else t[b:b + 1, :, h:h + 1]
        ref = oracle.backward(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["beta"]), sl(x["g"]),
                              None if x["h0"] is None else x["h0"][b:b + 1, h:h + 1],
                              sl(d_o), dhf[b:b + 1, h:h + 1])
        part = {n: (None if got[n] is None else (got[n][b:b + 1, :, h:h + 1] if n != "dh0"
                                                  else got[n][b:b + 1, h:h + 1]))
                for n in NAMES}
        stats = check(part, ref, f"head ({b},{h})")
        print("full size head", (b, h), {n: round(s["rel_max"], 8) for n, s in stats.items()})


def test_backward_directional_derivative_full_size(dp):
    """<grad, delta> for a random direction delta in every input equals the
    central difference of L = <d_o, o> + <dh_final, h_final> computed with
    the fp64 forward oracle (gated workload's recipe at B2 H4 T1024 n_h 4)."""
    w = W.GATED.scaled(B=2, H=4, T=1024)
    d_o, dhf = cotangents(w, 150)
    x = W.make_inputs(w)
    xc = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    got = dp.backward(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], xc["h0"], d_o=d_o.cuda(),
                      dh_final=dhf.cuda())
    gen = torch.Generator().manual_seed(151)
    xd = {k: x[k].double() for k in x if x[k] is not None}
    delta = {k: torch.randn(xd[k].shape, generator=gen, dtype=torch.float64) for k in xd}
    delta["g"] *= 0.01   # keep the gates inside (0, 1)
    grad_name = {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "g": "dg", "h0": "dh0"}
    lin = sum(float((got[grad_name[k]].cpu().double() * delta[k]).sum()) for k in xd)

    def loss(s):
        z = {k: xd[k] + s * delta[k] for k in xd}
        o, hf = oracle.forward(z["q"], z["k"], z["v"], z["beta"], z.get("g"), z.get("h0"))
        return float((torch.from_numpy(o) * d_o.double()).sum() + (torch.from_numpy(hf) * dhf.double()).sum())
    eps = 1e-4
    fd = (loss(eps) - loss(-eps)) / (2 * eps)
    print("directional derivative", lin, fd, abs(lin - fd) / abs(fd))
    assert abs(lin - fd) <= 1e-4 * abs(fd), (lin, fd)


def varlen_case(lengths, nh, seed, gated=True):
    T = int(sum(lengths))
    w = (W.GATED if gated else W.BASE).scaled(B=1, H=2, T=max(T, 1), nh=nh, seed=seed)
    x = W.make_inputs(w)
    pk = {k: (None if x[k] is None else x[k][0, :T].contiguous()) for k in ("q", "k", "v", "beta", "g")}
    gen = torch.Generator().manual_seed(seed + 1)
    N = len(lengths)
    pk["h0"] = 0.02 * torch.randn(N, 2, 128, 128, generator=gen)
    d_o = torch.randn(T, 2, 128, generator=gen)
    dhf = torch.randn(N, 2, 128, 128, generator=gen)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    return pk, d_o, dhf, cu


@pytest.mark.parametrize("gated,impl", [(True, "auto"), (True, "chunk_tc"), (False, "auto"), (False, "recurrent")],
                         ids=["gated-recurrent", "gated-chunked", "ungated-chunked", "ungated-recurrent"])
@pytest.mark.parametrize("lengths,nh", [([0, 1, 15, 30, 13], 2), ([40, 0, 7], 3), ([5], 1), ([17, 33], 4)])
def test_backward_varlen_parity(dp, lengths, nh, gated, impl):
    """Packed sequences: each sequence's gradients against the oracle's
    backward on that sequence alone, in both forms (the chunked one cuts
    each sequence into its own chunks)."""
    x, d_o, dhf, cu = varlen_case(lengths, nh, seed=60 + nh, gated=gated)
    xc = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    got, ws = dp.backward_varlen(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], xc["h0"], cu_seqlens=cu.cuda(),
                                 d_o=d_o.cuda(), dh_final=dhf.cuda(), impl=impl)
    dp.check_status(ws)
    a = 0
    for s, n in enumerate(lengths):
        sl = lambda t: None if t is None else t[a:a + n].unsqueeze(0)
        ref = oracle.backward(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["beta"]), sl(x["g"]), x["h0"][s:s + 1],
                              d_o[a:a + n].unsqueeze(0), dhf[s:s + 1])
        part = {nm: (got[nm][s:s + 1] if nm == "dh0" else (None if got[nm] is None else got[nm][a:a + n].unsqueeze(0)))
                for nm in NAMES}
        if n == 0:
            assert torch.equal(part["dh0"].cpu(), dhf[s:s + 1])
        else:
            check(part, ref, f"sequence {s} (length {n})")
        a += n


@pytest.mark.parametrize("gated", [True, False], ids=["recurrent", "chunked"])
def test_backward_varlen_bad_offsets(dp, gated):
    x, d_o, dhf, cu = varlen_case([20, 20], 2, seed=70, gated=gated)
    xc = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    bad = torch.tensor([0, 30, 20], dtype=torch.int32, device="cuda")
    _, ws = dp.backward_varlen(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], xc["h0"], cu_seqlens=bad,
                               max_seqlen=30, d_o=d_o.cuda(), dh_final=dhf.cuda())
    with pytest.raises(dp.DPError) as e:
        dp.check_status(ws)
    assert e.value.code == 7


def test_backward_chains_across_calls(dp):
    """A sequence cut in two: the second call starts from the first call's
    final state and hands its dh0 to the first call as dh_final; the
    gradients equal the single call's (the way a trainer carries state
    across segments)."""
    w = W.GATED.scaled(B=2, H=2, T=60, nh=2)
    d_o, dhf = cotangents(w, 160)
    x = W.make_inputs(w)
    xc = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    full = dp.backward(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], xc["h0"], d_o=d_o.cuda(), dh_final=dhf.cuda())
    t1 = 23
    part = lambda t, a, b: None if t is None else t[:, a:b].contiguous()
    xs1 = {k: part(xc[k], 0, t1) for k in ("q", "k", "v", "beta", "g")}
    xs2 = {k: part(xc[k], t1, w.T) for k in ("q", "k", "v", "beta", "g")}
    _, h_mid = dp.forward(xs1["q"], xs1["k"], xs1["v"], xs1["beta"], xs1["g"], xc["h0"], impl="recurrent",
                          out_dtype=torch.float32)
    g2 = dp.backward(xs2["q"], xs2["k"], xs2["v"], xs2["beta"], xs2["g"], h_mid, d_o=d_o[:, t1:].contiguous().cuda(),
                     dh_final=dhf.cuda())
    g1 = dp.backward(xs1["q"], xs1["k"], xs1["v"], xs1["beta"], xs1["g"], xc["h0"],
                     d_o=d_o[:, :t1].contiguous().cuda(), dh_final=g2["dh0"])
    for n in ("dq", "dk", "dv", "dbeta", "dg"):
        s = err_stats(torch.cat([g1[n], g2[n]], 1), full[n].cpu().double().numpy())
        assert s["rel_max"] <= TOL_REL, (n, s)
    s = err_stats(g1["dh0"], full["dh0"].cpu().double().numpy())
    assert s["rel_max"] <= TOL_REL, ("dh0", s)


# Ungated, D_k = D_v = 128: the chunked form (auto's choice) and the recurrent
# form, each against the oracle. Chunks hold min(16, 32 / n_h) tokens; the
# cases cut the sequence into several chunks with a ragged last one, a
# single exact chunk, one token, and both input dtypes.
CHUNK_CASES = [
    ("nh1-ragged", W.BASE.scaled(B=2, H=2, T=40, nh=1), 20),
    ("nh2-h0", W.BASE.scaled(B=1, H=2, T=37, h0_std=0.02), 21),
    ("nh3-neardup", W.NEARDUP.scaled(B=1, H=2, T=31), 22),
    ("nh4-beta2-h0", W.GATED.scaled(B=1, H=2, T=27, gated=False), 23),
    ("f32-nh2", W.BASE.scaled(B=1, H=1, T=20, dtype="f32"), 24),
    ("one-chunk", W.BASE.scaled(B=1, H=1, T=16), 25),
    ("one-token", W.BASE.scaled(B=2, H=1, T=1), 26),
]


@pytest.mark.parametrize("impl", ["chunk_tc", "recurrent"])
@pytest.mark.parametrize("name,w,seed", CHUNK_CASES, ids=[c[0] for c in CHUNK_CASES])
def test_backward_ungated_forms(dp, name, w, seed, impl):
    d_o, dhf = cotangents(w, 200 + seed)
    got, ref, _ = run_both(dp, w, d_o, dhf, impl=impl)
    stats = check(got, ref, f"{impl} {name}")
    print(impl, name, {n: round(s["rel_max"], 8) for n, s in stats.items()})


def test_backward_chunked_bf16_cotangent_and_empty(dp):
    w = W.BASE.scaled(B=1, H=2, T=45, nh=3)
    d_o, _ = cotangents(w, 230, torch.bfloat16)
    got, ref, _ = run_both(dp, w, d_o, None, impl="chunk_tc")
    check(got, ref, "chunked, bf16 d_o")
    w0 = W.BASE.scaled(B=2, H=2, T=0)
    d_o, dhf = cotangents(w0, 231)
    got, _, _ = run_both(dp, w0, d_o, dhf, impl="chunk_tc")
    assert torch.equal(got["dh0"].cpu(), dhf)


def test_backward_chunked_unsupported(dp):
    """The chunked form takes dense problems with D = 128 only."""
    w = W.TINY.scaled(B=1, H=1, T=8, nh=2, Dk=64, Dv=64)
    x = {k: (None if v is None else v.cuda()) for k, v in W.make_inputs(w).items()}
    with pytest.raises(dp.DPError) as e:
        dp.backward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], d_o=torch.zeros(1, 8, 1, 64, device="cuda"),
                    impl="chunk_tc")
    assert e.value.code == 2


# Gated, D = 128, chunked form (impl="chunk_tc"; "auto" keeps the recurrent
# form for gated problems): every gradient including dg against the oracle.
GATED_CHUNK_CASES = [
    ("nh1", W.GATED.scaled(B=1, H=2, T=40, nh=1), 40),
    ("nh2", W.GATED.scaled(B=2, H=1, T=37, nh=2), 41),
    ("nh3", W.GATED.scaled(B=1, H=2, T=31, nh=3), 42),
    ("nh4", W.GATED.scaled(B=1, H=2, T=27, nh=4), 43),
    ("f32-nh2", W.GATED.scaled(B=1, H=1, T=20, nh=2, dtype="f32"), 44),
    ("one-token", W.GATED.scaled(B=2, H=1, T=1, nh=2), 45),
]


@pytest.mark.parametrize("name,w,seed", GATED_CHUNK_CASES, ids=[c[0] for c in GATED_CHUNK_CASES])
def test_backward_gated_chunked(dp, name, w, seed):
    d_o, dhf = cotangents(w, 300 + seed)
    got, ref, _ = run_both(dp, w, d_o, dhf, impl="chunk_tc")
    stats = check(got, ref, f"gated chunked {name}")
    print("gated chunked", name, {n: round(s["rel_max"], 8) for n, s in stats.items()})


def test_backward_gated_chunked_zero_and_small_gates(dp):
    """Gates of exactly 0 (a reset inside a chunk) and tiny gates: the
    chunked form takes every decay and the gate gradient as range sums of
    log gates that skip the gate itself (no division by it), so dg stays the
    oracle's exact derivative."""
    w = W.GATED.scaled(B=1, H=2, T=45, nh=2)
    x = W.make_inputs(w)
    g = x["g"].float().clone()
    g[0, 5, 0] = 0.0
    g[0, 20, 1] = 0.0
    g[0, 21, 1] = 1e-6
    g[0, 33, 0] = 1e-3
    x["g"] = g.to(x["g"].dtype)
    d_o, dhf = cotangents(w, 350)
    xc = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    got = dp.backward(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], xc["h0"], d_o=d_o.cuda(), dh_final=dhf.cuda(),
                      impl="chunk_tc")
    ref = oracle.backward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], d_o, dhf)
    check(got, ref, "zero and small gates")


def test_backward_gated_chunked_negative_gate_reported(dp):
    w = W.GATED.scaled(B=1, H=1, T=20, nh=2)
    x = W.make_inputs(w)
    g = x["g"].float().clone()
    g[0, 7, 0] = -0.5
    x["g"] = g.to(x["g"].dtype)
    xc = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    dims = dp._lib.make_dims(1, 20, 1, 128, 128, 2, xc["q"].dtype, "chunk_tc", torch.float32)
    ws = torch.zeros(dp._lib.backward_workspace_size(dims), dtype=torch.uint8, device="cuda")
    dp.backward(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], xc["h0"], d_o=torch.zeros(1, 20, 1, 128, device="cuda"),
                impl="chunk_tc", workspace=ws)
    with pytest.raises(dp.DPError) as e:
        dp.check_status(ws)
    assert e.value.code == 7


def test_backward_auto_keeps_recurrent_for_gated(dp):
    """AUTO on a gated problem runs the recurrent form: its gradients equal
    impl="recurrent"'s up to the order of that kernel's fp32 atomics (the
    value-column CTAs of a head add their parts of dq, dk, dbeta and dg),
    compared at 1e-5 of RMS (two runs of the recurrent form have differed by
    1.1e-6)."""
    w = W.GATED.scaled(B=1, H=2, T=30, nh=2)
    d_o, dhf = cotangents(w, 360)
    got_auto, ref, _ = run_both(dp, w, d_o, dhf, impl="auto")
    got_rec, _, _ = run_both(dp, w, d_o, dhf, impl="recurrent")
    for n in NAMES:
        if ref[n] is not None:
            s = err_stats(got_auto[n], got_rec[n].cpu().double().numpy())
            assert s["rel_max"] <= 1e-5, (n, s)
