"""GPU parity of the prefill that continues from a decode state
(hla_prefill_continue): a prefill with a state, then a continuation, must give
the oracle's layer over the concatenated sequence (the continuation's rows and
the final state), and decoding afterwards must go on as if the whole sequence
had been one prefill.  Cases cover prefills shorter than the budget (ring not
full), continuations that cross the start of absorption, varlen batches, a
fresh state, two continuations in a row, the GLA variant, windows up to the
decode budget (8 + 888), the tensor-core path (bf16, d 128, GQA 2/4/8) and the
token-serial one."""
import numpy as np
import pytest
import torch

from linearized_attention_rope_gb300 import hla, synth
from gpu_cases import assert_close, oracle_cfg, params_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    from linearized_attention_rope_gb300 import build

    build.build()


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _args(x):
    return (x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["wq"], x["wk"], x["wv"], x["cu_seqlens"])


def _rows(x, key, n):
    cu = x["cu_seqlens"].tolist()
    return x[key][cu[n]:cu[n + 1]]


def _oracle(wl, parts, n, h, oracle, **kw):
    """Oracle over the concatenation of sequence n's rows in each input dict of `parts`."""
    d, kv = wl.head_dim, h // (wl.n_q_heads // wl.n_kv_heads)
    cat = lambda key, hh: np.concatenate([_np(_rows(x, key, n)[:, hh]) for x in parts])  # noqa: E731
    x0 = parts[0]
    job = dict(q=cat("q", h), k=cat("k", kv), v=cat("v", kv), g=cat("g", h), beta=cat("beta", h),
               lam=float(x0["lam"][h]), wq=_np(x0["wq"][h * d:(h + 1) * d]), wk=_np(x0["wk"][kv * d:(kv + 1) * d]),
               wv=_np(x0["wv"][kv * d:(kv + 1) * d]))
    return oracle.layer_units(oracle_cfg(wl, oracle, **kw), [job])[0]


def _inputs(wl, seqlens, seed):
    w = synth.small(wl.name, seqlens, n_q_heads=wl.n_q_heads, n_kv_heads=wl.n_kv_heads, head_dim=wl.head_dim,
                    dtype=wl.dtype, n_sinks=wl.n_sinks, window=wl.window, seed=seed)
    x = synth.make_inputs(w, "cuda")
    base = synth.make_inputs(wl, "cuda")  # same filters, lambda for every part
    for key in ("wq", "wk", "wv", "lam"):
        x[key] = base[key]
    return x


CASES = [
    # dtype, d, hq, hkv, n_sinks, window, first lengths, continuation lengths
    # bf16 d128 (tensor-core path): GQA 2, 8 and 4; windows of 24, 56, 120 and 888; contexts shorter than
    # the budget (no gap between sinks and window) and longer; continuations of 1 token to a few chunks
    ("bf16", 128, 4, 2, 8, 24, [10, 200, 0], [70, 5, 130]),
    ("bf16", 128, 8, 1, 8, 56, [300, 1000], [64, 700]),
    ("bf16", 128, 4, 1, 8, 120, [129, 2000, 0], [1, 300, 128]),
    ("bf16", 128, 2, 1, 8, 888, [1000, 50], [500, 900]),
    # contexts of 1 to 6 tokens: the first new tokens' conv taps reach positions before 0
    ("bf16", 128, 4, 2, 8, 24, [3, 5, 1, 6], [20, 9, 70, 2]),
    # sequences with no new tokens beside ones with many
    ("bf16", 128, 4, 2, 8, 24, [40, 90, 7], [0, 133, 0]),
    # forty sequences: many sequence starts inside one feature span
    ("bf16", 128, 4, 1, 8, 24, [5, 100] * 20, [7, 3] * 20),
    # token-serial path
    ("bf16", 64, 4, 1, 3, 40, [30, 100], [90, 1]),
    ("f32", 64, 2, 1, 8, 56, [512, 20], [100, 300]),
]


@pytest.mark.parametrize("dtype,d,hq,hkv,ns,W,first,second", CASES)
@pytest.mark.parametrize("gla", [False, True])
def test_prefill_then_continue_then_decode(oracle_mod, dtype, d, hq, hkv, ns, W, first, second, gla):
    flags = hla.FLAG_L2NORM_Q | (hla.FLAG_GLA if gla else 0)
    wl = synth.small(f"cont {dtype} d{d}", first, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, dtype=dtype,
                     n_sinks=ns, window=W, decode_steps=6)
    x1 = synth.make_inputs(wl, "cuda")
    x2 = _inputs(wl, second, synth.BASE_SEED + 321)
    prm = params_for(wl, flags)
    st = hla.State(prm, wl.n_seqs).init()
    out1 = torch.empty_like(x1["q"])
    hla.prefill(prm, *_args(x1), out1, state=st)
    out2 = torch.full_like(x2["q"], float("nan"))
    hla.prefill_continue(prm, *_args(x2), out2, st)
    # then a few decode steps
    douts = []
    for s in range(wl.decode_steps):
        o = torch.empty(x1["dq"].shape[1:], dtype=x1["dq"].dtype, device="cuda")
        hla.decode_step(prm, x1["dq"][s], x1["dk"][s], x1["dv"][s], x1["dg"][s], x1["dbeta"][s], x1["lam"], x1["wq"],
                        x1["wk"], x1["wv"], st, o)
        douts.append(o)
    torch.cuda.synchronize()
    assert st.check_error() == 0
    assert st.view("pos").cpu().tolist() == [a + b + wl.decode_steps for a, b in zip(first, second)]
    dec = {"q": x1["dq"], "k": x1["dk"], "v": x1["dv"], "g": x1["dg"], "beta": x1["dbeta"]}
    for n in range(wl.n_seqs):
        # decode tokens of sequence n as a third "part"
        x3 = {key: dec[key][:, n] for key in dec}
        x3["cu_seqlens"] = torch.tensor([0, wl.decode_steps], dtype=torch.int32, device="cuda")
        for h in range(hq):
            xs = [dict(x1, cu_seqlens=x1["cu_seqlens"]), x2]
            xn = [{k_: _rows(x, k_, n) for k_ in ("q", "k", "v", "g", "beta")} for x in xs]
            parts = []
            for xx in xn:
                xx = dict(xx)
                xx["cu_seqlens"] = torch.tensor([0, xx["q"].shape[0]], dtype=torch.int32, device="cuda")
                parts.append(xx)
            parts.append(x3)
            parts[0].update({k_: x1[k_] for k_ in ("wq", "wk", "wv", "lam")})
            ref = _oracle(wl, parts, 0, h, oracle_mod, erase_off=gla)
            a, b = first[n], first[n] + second[n]
            if second[n]:
                cu2 = x2["cu_seqlens"].tolist()
                got = _np(out2[cu2[n]:cu2[n + 1], h])
                assert_close(got, ref["o"][a:b], dtype, f"continuation rows seq {n} head {h}")
            got_dec = np.stack([_np(o[n, h]) for o in douts])
            assert_close(got_dec, ref["o"][b:], dtype, f"decode after continuation seq {n} head {h}")
            S = st.view("S").view(wl.n_seqs, hq, d, d)[n, h].cpu().numpy()
            assert_close(S, ref["S"], dtype, f"final S seq {n} head {h}")


def test_continue_from_a_fresh_state_equals_prefill(oracle_mod):
    wl = synth.small("cont fresh", [300, 64, 7], n_q_heads=4, n_kv_heads=2, head_dim=128)
    x = synth.make_inputs(wl, "cuda")
    prm = params_for(wl)
    st = hla.State(prm, wl.n_seqs).init()
    out = torch.empty_like(x["q"])
    hla.prefill_continue(prm, *_args(x), out, st)
    ref_out = torch.empty_like(x["q"])
    st_ref = hla.State(prm, wl.n_seqs).init()
    hla.prefill(prm, *_args(x), ref_out, state=st_ref)
    torch.cuda.synchronize()
    assert_close(out.float().cpu().numpy(), ref_out.float().cpu().numpy(), "bf16", "continue from pos 0")
    for name in ("S", "pend_k", "pend_v", "pend_g", "pend_beta", "conv_q", "conv_k", "conv_v"):
        assert_close(st.view(name).float().cpu().numpy(), st_ref.view(name).float().cpu().numpy(), "bf16", name)
    assert st.view("pos").cpu().tolist() == [300, 64, 7]


@pytest.mark.parametrize("d", [64, 128])
def test_two_continuations_in_a_row(oracle_mod, d):
    wl = synth.small("cont twice", [40], n_q_heads=2, n_kv_heads=1, head_dim=d, n_sinks=4, window=16)
    x1 = synth.make_inputs(wl, "cuda")
    x2 = _inputs(wl, [25], synth.BASE_SEED + 11)
    x3 = _inputs(wl, [33], synth.BASE_SEED + 12)
    prm = params_for(wl)
    st = hla.State(prm, 1).init()
    hla.prefill(prm, *_args(x1), torch.empty_like(x1["q"]), state=st)
    o2, o3 = torch.empty_like(x2["q"]), torch.empty_like(x3["q"])
    hla.prefill_continue(prm, *_args(x2), o2, st)
    hla.prefill_continue(prm, *_args(x3), o3, st)
    torch.cuda.synchronize()
    for h in range(2):
        parts = [x1, x2, x3]
        ref = _oracle(wl, parts, 0, h, oracle_mod)
        assert_close(_np(o2[:, h]), ref["o"][40:65], "bf16", f"second part head {h}")
        assert_close(_np(o3[:, h]), ref["o"][65:], "bf16", f"third part head {h}")
        assert_close(st.view("S").view(1, 2, d, d)[0, h].cpu().numpy(), ref["S"], "bf16", f"S head {h}")


def test_stale_workspace_contents_do_not_leak(oracle_mod):
    """The same calls with a workspace full of non-finite bytes give the same bits as with a zeroed one: the
    tensor-core kernels read whole tiles past a sequence's end, and those rows must be written or zeroed."""
    wl = synth.small("cont stale", [300, 50], n_q_heads=4, n_kv_heads=1, head_dim=128, n_sinks=8, window=56)
    x1 = synth.make_inputs(wl, "cuda")
    x2 = _inputs(wl, [130, 7], synth.BASE_SEED + 33)
    prm = params_for(wl)
    outs = []
    for fill in (0x00, 0xFF):
        st = hla.State(prm, wl.n_seqs).init()
        ws1 = torch.full((hla.workspace_bytes(prm, x1["q"].shape[0], wl.n_seqs),), fill, dtype=torch.uint8,
                         device="cuda")
        o1 = torch.empty_like(x1["q"])
        hla.prefill(prm, *_args(x1), o1, state=st, ws=ws1)
        ws2 = torch.full((hla.continue_workspace_bytes(prm, x2["q"].shape[0], wl.n_seqs),), fill, dtype=torch.uint8,
                         device="cuda")
        o2 = torch.empty_like(x2["q"])
        hla.prefill_continue(prm, *_args(x2), o2, st, ws=ws2)
        torch.cuda.synchronize()
        outs.append((o1.clone(), o2.clone(), st.view("S").clone()))
    for a, b in zip(*outs):
        assert torch.isfinite(b.float()).all()
        assert torch.equal(a, b)


@pytest.mark.parametrize("d", [64, 128])
def test_negative_position_is_flagged_and_left_alone(d):
    wl = synth.small("cont neg", [100, 80], n_q_heads=4, n_kv_heads=2, head_dim=d)
    x1 = synth.make_inputs(wl, "cuda")
    x2 = _inputs(wl, [30, 20], synth.BASE_SEED + 44)
    prm = params_for(wl)
    st = hla.State(prm, 2).init()
    hla.prefill(prm, *_args(x1), torch.empty_like(x1["q"]), state=st)
    torch.cuda.synchronize()
    st.view("pos")[1] = -5  # a position no prefill or decode step leaves
    before = {name: st.view(name)[:].clone() for name in ("S", "k_ring", "conv_k")}
    hla.prefill_continue(prm, *_args(x2), torch.empty_like(x2["q"]), st)
    torch.cuda.synchronize()
    assert st.check_error() != 0
    assert st.view("pos").cpu().tolist() == [130, -5]
    half = lambda t: t.view(2, -1)[1]  # noqa: E731  sequence 1's part of a per-sequence buffer
    for name, b in before.items():
        assert torch.equal(half(st.view(name)), half(b)), name


def test_continue_layer_shape_wide_spans(oracle_mod):
    # the LLaMA-3.1-8B layer shape (32 q-heads, 8 kv-heads) with about 4,200 new tokens: the feature kernel's
    # token spans are then many steps long (one wave of CTAs), and steps cross sequence starts inside a span
    first, second = [600, 3000, 5], [2500, 1700, 13]
    wl = synth.small("cont wide", first, n_q_heads=32, n_kv_heads=8, head_dim=128)
    x1 = synth.make_inputs(wl, "cuda")
    x2 = _inputs(wl, second, synth.BASE_SEED + 45)
    prm = params_for(wl)
    st = hla.State(prm, 3).init()
    hla.prefill(prm, *_args(x1), torch.empty_like(x1["q"]), state=st)
    out2 = torch.full_like(x2["q"], float("nan"))
    hla.prefill_continue(prm, *_args(x2), out2, st)
    # every head: the same sequences in one prefill
    xw = {key: torch.cat([torch.cat([_rows(x1, key, n), _rows(x2, key, n)]) for n in range(3)])
          for key in ("q", "k", "v", "g", "beta")}
    xw.update({key: x1[key] for key in ("wq", "wk", "wv", "lam")})
    lens = [a + b for a, b in zip(first, second)]
    xw["cu_seqlens"] = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    st_w = hla.State(prm, 3).init()
    out_w = torch.empty_like(xw["q"])
    hla.prefill(prm, *_args(xw), out_w, state=st_w)
    torch.cuda.synchronize()
    assert st.check_error() == 0
    cw, c2 = xw["cu_seqlens"].tolist(), x2["cu_seqlens"].tolist()
    for n in range(3):
        assert_close(_np(out2[c2[n]:c2[n + 1]]), _np(out_w[cw[n] + first[n]:cw[n + 1]]), "bf16", f"seq {n} vs one prefill")
    for name in ("S", "k_ring", "v_ring", "conv_q", "conv_k", "conv_v"):
        assert_close(st.view(name).float().cpu().numpy(), st_w.view(name).float().cpu().numpy(), "bf16", name)
    # the pending ring on its live slots (the tokens still waiting; the slot of the token absorbed last is
    # never read again and keeps whatever the earlier call left there)
    P = wl.window + 1
    for name, heads in (("pend_k", 8), ("pend_v", 8), ("pend_g", 32), ("pend_beta", 32)):
        a = st.view(name).float().cpu().numpy().reshape(3, heads, P, -1)
        b = st_w.view(name).float().cpu().numpy().reshape(3, heads, P, -1)
        for n, L in enumerate(lens):
            live = [p % P for p in range(max(L - wl.window, wl.n_sinks), L)]
            assert_close(a[n][:, live], b[n][:, live], "bf16", f"{name} seq {n}")
    # sampled heads (three kv groups) against the oracle
    for n in (0, 1):
        for h in (0, 13, 31):
            ref = _oracle(wl, [x1, x2], n, h, oracle_mod)
            assert_close(_np(out2[c2[n]:c2[n + 1], h]), ref["o"][first[n]:], "bf16", f"seq {n} head {h}")
            S = st.view("S").view(3, 32, 128, 128)[n, h].cpu().numpy()
            assert_close(S, ref["S"], "bf16", f"S seq {n} head {h}")


def test_overlapping_sequences_are_flagged():
    # sequences 0 and 2 overlap (cu not monotone): their extended rows would add up past the workspace's
    # bound, so the table is flagged and every row stays inside the workspace
    wl = synth.small("cont overlap", [100, 80, 60], n_q_heads=4, n_kv_heads=2, head_dim=128)
    x1 = synth.make_inputs(wl, "cuda")
    x2 = _inputs(wl, [45, 0, 5], synth.BASE_SEED + 46)
    x2["cu_seqlens"] = torch.tensor([0, 45, 5, 50], dtype=torch.int32, device="cuda")
    prm = params_for(wl)
    st = hla.State(prm, 3).init()
    hla.prefill(prm, *_args(x1), torch.empty_like(x1["q"]), state=st)
    hla.prefill_continue(prm, *_args(x2), torch.empty_like(x2["q"]), st)
    torch.cuda.synchronize()
    assert st.check_error() == 1  # the sequence-table error
