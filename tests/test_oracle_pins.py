"""Pins for the fp64 CPU oracle: each checks it against something other than
itself -- a library routine on a special case (torch fp64 SDPA and autograd
per segment), closed forms, central finite differences, exact gradient
invariants, and the values the pages print.  A final test plants plausible
mistakes into copies of the oracle source and checks that this battery
catches every one.
"""
import json
import math
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from packed_variable_length_varlen_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_values.json")


def _cu(lens):
    return [0] + list(np.cumsum(lens).astype(int))


def _rand(shape, seed, dtype=torch.float64, amp=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g, dtype=torch.float64) * amp).to(dtype)


def _problem(lq, lk, H, D, seed=0, dtype=torch.float64, amp=1.0, scale=None, strided=False):
    cq, ck = _cu(lq), _cu(lk)
    if strided:  # padded row stride, NaN in the padding
        def mk(n, s):
            buf = torch.full((n, H * D + 24), float("nan"), dtype=dtype)
            t = buf[:, :H * D].unflatten(1, (H, D))
            t.copy_(_rand((n, H, D), s, dtype, amp))
            return t
    else:
        def mk(n, s):
            return _rand((n, H, D), s, dtype, amp)
    q, k, v = mk(cq[-1], seed), mk(ck[-1], seed + 1), mk(ck[-1], seed + 2)
    do = mk(cq[-1], seed + 3)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    return oracle.Problem(q, k, v, cq, ck, scale, dout=do), (q, k, v, do, cq, ck, scale)


def _torch_reference(q, k, v, do, cq, ck, scale):
    """Per segment: torch fp64 SDPA forward, logsumexp, and autograd."""
    H, D = q.shape[1], q.shape[2]
    out = torch.zeros(q.shape, dtype=torch.float64)
    lse = torch.full((q.shape[0], H), float("nan"), dtype=torch.float64)
    dq = torch.zeros(q.shape, dtype=torch.float64)
    dk = torch.zeros(k.shape, dtype=torch.float64)
    dv = torch.zeros(v.shape, dtype=torch.float64)
    for b in range(len(cq) - 1):
        qs = q[cq[b]:cq[b + 1]].double().transpose(0, 1).clone().requires_grad_()
        ks = k[ck[b]:ck[b + 1]].double().transpose(0, 1).clone().requires_grad_()
        vs = v[ck[b]:ck[b + 1]].double().transpose(0, 1).clone().requires_grad_()
        if qs.shape[1] == 0 or ks.shape[1] == 0:
            continue  # empty sums: covered by the closed-form tests
        o = F.scaled_dot_product_attention(qs[None], ks[None], vs[None], scale=scale)[0]
        gq, gk, gv = torch.autograd.grad(o, (qs, ks, vs), do[cq[b]:cq[b + 1]].double().transpose(0, 1))
        out[cq[b]:cq[b + 1]] = o.detach().transpose(0, 1)
        lse[cq[b]:cq[b + 1]] = torch.logsumexp(scale * (qs @ ks.transpose(1, 2)), dim=-1).detach().T
        dq[cq[b]:cq[b + 1]] = gq.transpose(0, 1)
        dk[ck[b]:ck[b + 1]] = gk.transpose(0, 1)
        dv[ck[b]:ck[b + 1]] = gv.transpose(0, 1)
    return out, lse, dq, dk, dv


def _torch_causal_reference(q, k, v, do, cq, ck, scale):
    """Per segment, causal: masked softmax attention in fp64 torch ops with
    the mask of the reading (key jj visible to query ii iff
    jj <= ii + Sk - Sq), gradients by autograd; a row that sees no key gets
    o = 0 and LSE = -inf."""
    H, D = q.shape[1], q.shape[2]
    out = torch.zeros(q.shape, dtype=torch.float64)
    lse = torch.full((q.shape[0], H), float("-inf"), dtype=torch.float64)
    dq = torch.zeros(q.shape, dtype=torch.float64)
    dk = torch.zeros(k.shape, dtype=torch.float64)
    dv = torch.zeros(v.shape, dtype=torch.float64)
    for b in range(len(cq) - 1):
        Sq, Sk = cq[b + 1] - cq[b], ck[b + 1] - ck[b]
        if Sq == 0 or Sk == 0:
            continue
        qs = q[cq[b]:cq[b + 1]].double().transpose(0, 1).clone().requires_grad_()
        ks = k[ck[b]:ck[b + 1]].double().transpose(0, 1).clone().requires_grad_()
        vs = v[ck[b]:ck[b + 1]].double().transpose(0, 1).clone().requires_grad_()
        vis = torch.arange(Sk)[None, :] <= torch.arange(Sq)[:, None] + (Sk - Sq)   # [Sq, Sk]
        live = vis.any(-1)                                                        # [Sq]
        s = scale * (qs @ ks.transpose(1, 2))
        s = torch.where(vis, s, torch.full_like(s, float("-inf")))
        s = torch.where(live[:, None], s, torch.zeros_like(s))   # dead rows: no NaN in the graph
        p = torch.where(live[:, None], torch.softmax(s, -1), torch.zeros_like(s))
        o = p @ vs
        gq, gk, gv = torch.autograd.grad(o, (qs, ks, vs), do[cq[b]:cq[b + 1]].double().transpose(0, 1))
        out[cq[b]:cq[b + 1]] = o.detach().transpose(0, 1)
        l = torch.logsumexp(s.detach(), dim=-1)
        lse[cq[b]:cq[b + 1]] = torch.where(live[None, :], l, torch.full_like(l, float("-inf"))).T
        dq[cq[b]:cq[b + 1]] = gq.transpose(0, 1)
        dk[ck[b]:ck[b + 1]] = gk.transpose(0, 1)
        dv[ck[b]:ck[b + 1]] = gv.transpose(0, 1)
    return out, lse, dq, dk, dv


def _causal_checks(lib, seed):
    """Causal-mask pins: the masked torch reference, fp64 SDPA with
    is_causal on the equal-length segment, rows that see no key, and rows
    that see every key (identical to the unmasked oracle)."""
    res = []
    lq, lk = [5, 9, 6, 1, 0, 4], [9, 4, 6, 3, 2, 0]  # Sq < Sk, Sq > Sk (dead rows), Sq = Sk, one row, empties
    H, D = 2, 8
    cq, ck = _cu(lq), _cu(lk)
    q, k, v = _rand((cq[-1], H, D), seed + 30), _rand((ck[-1], H, D), seed + 31), _rand((ck[-1], H, D), seed + 32)
    do = _rand((cq[-1], H, D), seed + 33)
    sc = 0.37
    pc = oracle.Problem(q, k, v, cq, ck, sc, dout=do, causal=True)
    pn = oracle.Problem(q, k, v, cq, ck, sc, dout=do)
    rows, heads = oracle.all_pairs(cq[-1], H)
    krows, kheads = oracle.all_pairs(ck[-1], H)
    o, lse = pc.fwd(rows, heads, lib=lib)
    dq, _ = pc.bwd_q(rows, heads, lib=lib)
    dk, dv = pc.bwd_kv(krows, kheads, lib=lib)
    ro, rl, rdq, rdk, rdv = _torch_causal_reference(q, k, v, do, cq, ck, sc)
    res.append(("causal_out", np.allclose(o, ro.reshape(-1, D).numpy(), rtol=1e-12, atol=1e-13)))
    res.append(("causal_lse", np.allclose(lse, rl.reshape(-1).numpy(), rtol=1e-12, atol=1e-13)))
    res.append(("causal_dq", np.allclose(dq, rdq.reshape(-1, D).numpy(), rtol=1e-10, atol=1e-12)))
    res.append(("causal_dk", np.allclose(dk, rdk.reshape(-1, D).numpy(), rtol=1e-10, atol=1e-12)))
    res.append(("causal_dv", np.allclose(dv, rdv.reshape(-1, D).numpy(), rtol=1e-10, atol=1e-12)))
    # equal lengths: fp64 SDPA with is_causal (a library routine)
    b = 2
    qs, ks, vs = (t[c[b]:c[b + 1]].transpose(0, 1)[None] for t, c in ((q, cq), (k, ck), (v, ck)))
    so = F.scaled_dot_product_attention(qs, ks, vs, scale=sc, is_causal=True)[0].transpose(0, 1)
    sel = (rows >= cq[b]) & (rows < cq[b + 1])
    res.append(("causal_sdpa_is_causal", np.allclose(o[sel], so.reshape(-1, D).numpy(), rtol=1e-12, atol=1e-13)))
    # rows that see no key: segment 1 (Sq=9, Sk=4), rows 0..4
    dead = (rows >= cq[1]) & (rows < cq[1] + 5)
    res.append(("causal_dead_rows", bool(np.all(np.isneginf(lse[dead])) and np.all(o[dead] == 0)
                                         and np.all(dq[dead] == 0))))
    # the last row of every segment with keys sees them all: same numbers as unmasked
    on, ln = pn.fwd(rows, heads, lib=lib)
    last = np.zeros(rows.shape, bool)
    for bb in range(len(lq)):
        if lq[bb] > 0 and lk[bb] > 0:
            last |= rows == cq[bb + 1] - 1
    res.append(("causal_last_row_unmasked", bool(np.array_equal(o[last], on[last]) and np.array_equal(lse[last], ln[last]))))
    # Sq = Sk: the first row sees only the first key -> o = v_0
    first = rows == cq[2]
    res.append(("causal_first_row_v0", bool(np.array_equal(o[first], v[ck[2]].numpy()))))
    return res


def _all(pb, total):
    return oracle.all_pairs(total, pb.H)


# lengths: include empty q, empty k, one-key, Sq != Sk, multi-row segments
LQ = [5, 0, 3, 1, 17, 6, 9]
LK = [7, 4, 1, 1, 23, 6, 0]


def _battery(lib, seed=0):
    """The pin checks as a list of (name, ok) so that planted-mistake builds
    can run all of them.  Uses only torch / numpy / closed forms."""
    res = []
    H, D = 2, 8
    pb, (q, k, v, do, cq, ck, sc) = _problem(LQ, LK, H, D, seed=seed)
    ro, rl, rdq, rdk, rdv = _torch_reference(q, k, v, do, cq, ck, sc)
    rows, heads = _all(pb, cq[-1])
    o, lse = pb.fwd(rows, heads, lib=lib)
    dq, _ = pb.bwd_q(rows, heads, lib=lib)
    krows, kheads = _all(pb, ck[-1])
    dk, dv = pb.bwd_kv(krows, kheads, lib=lib)
    # rows whose segment has keys
    has_k = np.zeros(cq[-1], bool)
    for b in range(len(LQ)):
        has_k[cq[b]:cq[b + 1]] = LK[b] > 0
    m = np.repeat(has_k, H)
    res.append(("sdpa_out", np.allclose(o[m], ro.reshape(-1, D).numpy()[m], rtol=1e-12, atol=1e-13)))
    res.append(("sdpa_lse", np.allclose(lse[m], rl.reshape(-1).numpy()[m], rtol=1e-12, atol=1e-13)))
    res.append(("autograd_dq", np.allclose(dq[m], rdq.reshape(-1, D).numpy()[m], rtol=1e-10, atol=1e-12)))
    has_q = np.zeros(ck[-1], bool)
    for b in range(len(LQ)):
        has_q[ck[b]:ck[b + 1]] = LQ[b] > 0
    mk_ = np.repeat(has_q, H)
    res.append(("autograd_dk", np.allclose(dk[mk_], rdk.reshape(-1, D).numpy()[mk_], rtol=1e-10, atol=1e-12)))
    res.append(("autograd_dv", np.allclose(dv[mk_], rdv.reshape(-1, D).numpy()[mk_], rtol=1e-10, atol=1e-12)))
    # empty-key rows: LSE -inf, O = 0, dQ = 0; empty-query kv rows: dK = dV = 0
    res.append(("empty_k", bool(np.all(np.isneginf(lse[~m])) and np.all(o[~m] == 0) and np.all(dq[~m] == 0))))
    res.append(("empty_q", bool(np.all(dk[~mk_] == 0) and np.all(dv[~mk_] == 0))))
    # closed form: Q = 0 -> O = mean V, LSE = ln Sk, dv_j = mean_i dO_i
    qz = torch.zeros_like(q)
    pz = oracle.Problem(qz, k, v, cq, ck, sc, dout=do)
    oz, lz = pz.fwd(rows, heads, lib=lib)
    dkz, dvz = pz.bwd_kv(krows, kheads, lib=lib)
    ok_o = ok_l = ok_dv = True
    for b in range(len(LQ)):
        if LQ[b] == 0 or LK[b] == 0:
            continue
        vm = v[ck[b]:ck[b + 1]].mean(0).numpy()          # [H, D]
        dom = do[cq[b]:cq[b + 1]].sum(0).numpy() / LK[b]  # [H, D]
        sel = (rows >= cq[b]) & (rows < cq[b + 1])
        ok_o &= np.allclose(oz[sel], vm[heads[sel]], rtol=1e-13, atol=1e-14)
        ok_l &= np.allclose(lz[sel], math.log(LK[b]), rtol=1e-14, atol=1e-14)
        kse = (krows >= ck[b]) & (krows < ck[b + 1])
        ok_dv &= np.allclose(dvz[kse], dom[kheads[kse]], rtol=1e-12, atol=1e-13)
    res += [("qzero_mean_v", ok_o), ("qzero_lse_lnSk", ok_l), ("qzero_dv", ok_dv)]
    # closed form: one-key segment (segment 3: Sq=1, Sk=1) -> o = v, LSE = scale q.k, dq = dk = 0
    b = 3
    i, j = cq[b], ck[b]
    sel = rows == i
    ksel = krows == j
    ok1 = np.allclose(o[sel], v[j].numpy(), rtol=0, atol=1e-15)
    ok2 = np.allclose(lse[sel], sc * (q[i] * k[j]).sum(-1).numpy(), rtol=1e-13, atol=1e-14)
    ok3 = np.allclose(dq[sel], 0, atol=1e-15) and np.allclose(dk[ksel], 0, atol=1e-15)
    res += [("onekey_o", ok1), ("onekey_lse", ok2), ("onekey_grads_zero", ok3)]
    # closed form: one-hot V exposes P: rows sum to 1, ratios are exp(s_ij - s_ik)
    Dh = 24
    lq2, lk2 = [4, 3], [5, 24]
    cq2, ck2 = _cu(lq2), _cu(lk2)
    q2 = _rand((cq2[-1], 1, Dh), seed + 9)
    k2 = _rand((ck2[-1], 1, Dh), seed + 10)
    v2 = torch.zeros(ck2[-1], 1, Dh, dtype=torch.float64)
    for b2 in range(2):
        for jj in range(lk2[b2]):
            v2[ck2[b2] + jj, 0, jj] = 1.0
    p2 = oracle.Problem(q2, k2, v2, cq2, ck2, 0.3)
    r2, h2 = oracle.all_pairs(cq2[-1], 1)
    P, _ = p2.fwd(r2, h2, lib=lib)
    okp = np.allclose(P.sum(1), 1.0, rtol=0, atol=1e-14)
    for b2 in range(2):
        for ii in range(cq2[b2], cq2[b2 + 1]):
            s = 0.3 * (k2[ck2[b2]:ck2[b2 + 1], 0] @ q2[ii, 0]).numpy()
            okp &= np.allclose(P[ii, :lk2[b2]] / P[ii, 0], np.exp(s - s[0]), rtol=1e-12)
            okp &= np.all(P[ii, lk2[b2]:] == 0)
    res.append(("onehot_v_softmax", bool(okp)))
    # closed form: constant V -> constant O
    vc = torch.full_like(v, 0.75)
    pc = oracle.Problem(q, k, vc, cq, ck, sc)
    oc, _ = pc.fwd(rows, heads, lib=lib)
    res.append(("const_v", bool(np.allclose(oc[m], 0.75, rtol=0, atol=1e-14))))
    # shift invariance: k_j -> k_j + u moves LSE_i by scale q_i.u, O unchanged
    u = _rand((1, H, D), seed + 11)
    ps = oracle.Problem(q, k + u, v, cq, ck, sc)
    os_, ls_ = ps.fwd(rows, heads, lib=lib)
    shift = sc * (q * u).sum(-1).reshape(-1).numpy()
    res.append(("shift_o", bool(np.allclose(os_[m], o[m], rtol=1e-11, atol=1e-12))))
    res.append(("shift_lse", bool(np.allclose(ls_[m], lse[m] + shift[m], rtol=1e-11, atol=1e-12))))
    # gradient invariants per (segment, head): sum_j dk_j = 0, sum_j dv_j = sum_i dO_i
    inv = True
    for b in range(len(LQ)):
        if LQ[b] == 0 or LK[b] == 0:
            continue
        kse = (krows >= ck[b]) & (krows < ck[b + 1])
        for h in range(H):
            sh = kse & (kheads == h)
            inv &= np.allclose(dk[sh].sum(0), 0, atol=1e-12)
            inv &= np.allclose(dv[sh].sum(0), do[cq[b]:cq[b + 1], h].sum(0).numpy(), atol=1e-12)
    res.append(("grad_invariants", bool(inv)))
    # central finite differences of L = sum(O * dO)
    res.append(("finite_differences", _finite_difference_ok(lib, seed)))
    res += _causal_checks(lib, seed)
    return res


def _finite_difference_ok(lib, seed, h=1e-5):
    lq, lk = [3, 0, 1, 4], [2, 3, 1, 5]
    H, D = 1, 6
    pb, (q, k, v, do, cq, ck, sc) = _problem(lq, lk, H, D, seed=seed + 20)
    rows, heads = oracle.all_pairs(cq[-1], H)
    krows, kheads = oracle.all_pairs(ck[-1], H)
    dq, _ = pb.bwd_q(rows, heads, lib=lib)
    dk, dv = pb.bwd_kv(krows, kheads, lib=lib)
    dvec = do.reshape(-1, D).numpy()

    def loss(qq, kk, vv):
        p = oracle.Problem(qq, kk, vv, cq, ck, sc)
        o, _ = p.fwd(rows, heads, lib=lib)
        return float((o * dvec).sum())

    ok = True
    for name, base, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        flat = base.reshape(-1)
        num = np.zeros(flat.numel())
        for e in range(flat.numel()):
            old = flat[e].item()
            flat[e] = old + h
            args = {"q": q, "k": k, "v": v}
            lp = loss(args["q"], args["k"], args["v"])
            flat[e] = old - h
            lm = loss(args["q"], args["k"], args["v"])
            flat[e] = old
            num[e] = (lp - lm) / (2 * h)
        ok &= np.allclose(grad.reshape(-1), num, rtol=1e-6, atol=1e-8)
    return bool(ok)


def test_oracle_battery(oracle_lib):
    res = _battery(oracle_lib)
    bad = [n for n, ok in res if not ok]
    assert not bad, "oracle pins failed: %s" % bad


def test_oracle_bf16_strided_matches_sdpa(oracle_lib):
    """bf16 inputs through padded (NaN-filled) row strides: widened exactly,
    padding never read."""
    H, D = 3, 16
    pb, (q, k, v, do, cq, ck, sc) = _problem([9, 4, 0, 31], [9, 13, 2, 31], H, D, seed=5,
                                             dtype=torch.bfloat16, strided=True)
    ro, rl, rdq, rdk, rdv = _torch_reference(q.double(), k.double(), v.double(), do.double(), cq, ck, sc)
    rows, heads = oracle.all_pairs(cq[-1], H)
    o, lse = pb.fwd(rows, heads)
    dq, _ = pb.bwd_q(rows, heads)
    krows, kheads = oracle.all_pairs(ck[-1], H)
    dk, dv = pb.bwd_kv(krows, kheads)
    assert np.isfinite(o).all() and np.isfinite(dq).all() and np.isfinite(dk).all()
    np.testing.assert_allclose(o, ro.reshape(-1, D).numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, rl.reshape(-1).numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dq, rdq.reshape(-1, D).numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, rdk.reshape(-1, D).numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, rdv.reshape(-1, D).numpy(), rtol=1e-10, atol=1e-12)


def test_oracle_pairs_subset_consistent(oracle_lib):
    """A sampled subset of pairs gives the same numbers as the full sweep."""
    H, D = 4, 8
    pb, (q, k, v, do, cq, ck, sc) = _problem([50, 70], [60, 40], H, D, seed=3)
    rows, heads = oracle.all_pairs(cq[-1], H)
    o, lse = pb.fwd(rows, heads)
    sel = np.array([0, 7, 13, 200, 479])
    o2, l2 = pb.fwd(rows[sel], heads[sel])
    assert np.array_equal(o2, o[sel]) and np.array_equal(l2, lse[sel])


def test_page_values():
    """Numbers printed on the pages: the int32 wrap of the dout offset and
    the exact per-segment tile count of the windowed workload."""
    g = json.load(open(GOLDEN))
    w = g["dout_offset_wrap"]
    true = w["coord"] * w["dout_stride"][0]
    assert true == w["true_offset"]
    wrapped = np.array([true], dtype=np.int64).astype(np.int32)[0]
    assert int(wrapped) == w["off_signed_i32"]
    assert int(np.array([wrapped], dtype=np.int64).view(np.uint64)[0]) == w["off_unsigned_i64"]
    t = g["dout_wrap_threshold"]
    assert t["num_heads"] * t["head_dim"] + t["mlp_dim"] == t["stride0"]
    assert abs(2 ** 31 / t["stride0"] - t["threshold_rows_approx"]) < 1.0
    assert W.offset_crossing_row(t["stride0"], 1) == t["threshold_rows_approx"]
    c = g["windowed_tile_count"]
    wl = W.windowed()
    assert list(wl.cu_q) == c["cu_seqlens_q"] and wl.num_heads == c["num_heads"]
    assert wl.q_tiles(c["tile_m"]) == c["valid_tiles"]
    assert max(wl.seqlens_q()) == c["true_max_seqlen_q"] != c["stated_max_seqlen_q"]


MUTANTS = [
    ("dropped scale in s", "s[j] = pb->scale * dot(qi, kj, D);", "s[j] = dot(qi, kj, D);"),
    ("LSE without the max", "const double lse = m + log(sum);", "const double lse = log(sum);"),
    ("exp of s without the max", "sum += exp(s[j] - m);", "sum += exp(s[j]);"),
    ("o sums K instead of V",
     "load_row(pb->v, pb->dtype, pb->v_rs, pb->v_hs, k0 + j, h, D, kj);\n        for (int32_t d = 0; d < D; ++d) out_o[d] += p * kj[d];",
     "load_row(pb->k, pb->dtype, pb->k_rs, pb->k_hs, k0 + j, h, D, kj);\n        for (int32_t d = 0; d < D; ++d) out_o[d] += p * kj[d];"),
    ("wrong sign in dS (q side)", "const double ds = p * (dp - dlt);", "const double ds = p * (dp + dlt);"),
    ("dV sums dS instead of P", "gv[d] += p * doi[d];", "gv[d] += ds * doi[d];"),
    ("dK misses the scale", "gk[d] += pb->scale * ds * qi[d];", "gk[d] += ds * qi[d];"),
    ("dK sums dO instead of Q", "gk[d] += pb->scale * ds * qi[d];", "gk[d] += pb->scale * ds * doi[d];"),
    ("segment end off by one", "if ((int64_t)cu[b] <= i && i < (int64_t)cu[b + 1]) return b;",
     "if ((int64_t)cu[b] <= i && i <= (int64_t)cu[b + 1]) return b;"),
    ("kv segment start of the next segment", "const int64_t k0 = pb->cu_k[b], Sk",
     "const int64_t k0 = pb->cu_k[b] + (b > 0), Sk"),
    ("delta from dO.v instead of dO.o", "E[ii] = dot(doi, oi, D);", "E[ii] = dot(doi, doi, D);"),
    ("head stride ignored", "int64_t off = row * rs + (int64_t)h * hs;", "int64_t off = row * rs;"),
    ("causal diagonal one key early", "const int64_t n = ii + (Sk - Sq) + 1;", "const int64_t n = ii + (Sk - Sq);"),
    ("causal diagonal aligned top-left", "const int64_t n = ii + (Sk - Sq) + 1;", "const int64_t n = ii + 1;"),
    ("causal mask missing on the key side", "if (jj >= visible_keys(pb, b, ii)) continue;", "(void)jj;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(oracle._SRC).read()
    assert src.count(old) >= 1, "mutation anchor missing: %s" % name
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    lib_path = str(tmp_path / "libmutant.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-shared", "-fPIC", "-o", lib_path,
                    str(mut), "-lm"], check=True)
    lib = oracle.load_library(lib_path)
    try:
        res = _battery(lib)
    except Exception:  # a crash or NaN blow-up also counts as caught
        return
    assert any(not ok for _, ok in res), "planted mistake '%s' not caught" % name
