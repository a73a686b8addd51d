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
import pathlib
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
    """Per segment, causal: the masked reference with key jj visible to
    query ii iff jj <= ii + Sk - Sq."""
    return _torch_masked_reference(q, k, v, do, cq, ck, scale, lambda i, j, d: j <= i + d)


def _torch_masked_reference(q, k, v, do, cq, ck, scale, visible):
    """Per segment: masked softmax attention in fp64 torch ops, key jj
    visible to query ii iff visible(ii, jj, Sk - Sq) (broadcast index
    tensors), gradients by autograd; a row that sees no key gets o = 0 and
    LSE = -inf."""
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
        vis = visible(torch.arange(Sq)[:, None], torch.arange(Sk)[None, :], Sk - Sq)   # [Sq, Sk]
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


def _window_checks(lib, seed):
    """Sliding-window pins: closed forms that fix each side of the band
    exactly (a zero-width band gives o_i = v of the diagonal key; a band of
    two keys is a two-term softmax), windows wider than every segment equal
    the unmasked oracle, (-1, 0) equals the causal mask, and the masked torch
    autograd reference for the gradients."""
    res = []
    H, D, sc = 2, 8, 0.41
    lq, lk = [7, 5, 9, 1, 0, 6], [7, 9, 4, 3, 2, 0]  # Sq = Sk, Sq < Sk, Sq > Sk, one row, empties
    cq, ck = _cu(lq), _cu(lk)
    q, k, v = _rand((cq[-1], H, D), seed + 40), _rand((ck[-1], H, D), seed + 41), _rand((ck[-1], H, D), seed + 42)
    do = _rand((cq[-1], H, D), seed + 43)
    rows, heads = oracle.all_pairs(cq[-1], H)
    krows, kheads = oracle.all_pairs(ck[-1], H)

    def run(**kw):
        pb = oracle.Problem(q, k, v, cq, ck, sc, dout=do, **kw)
        o, lse = pb.fwd(rows, heads, lib=lib)
        dq, _ = pb.bwd_q(rows, heads, lib=lib)
        dk, dv = pb.bwd_kv(krows, kheads, lib=lib)
        return o, lse, dq, dk, dv

    # zero-width band: q row ii sees only key ii + Sk - Sq (when it exists)
    o, lse, dq, dk, dv = run(window=(0, 0))
    ok0 = True
    for b in range(len(lq)):
        for ii in range(lq[b]):
            r = cq[b] + ii
            jj = ii + lk[b] - lq[b]
            for h in range(H):
                t = r * H + h
                if 0 <= jj < lk[b]:
                    kr = ck[b] + jj
                    s_exp = sc * float(torch.dot(q[r, h], k[kr, h]))
                    ok0 &= bool(np.array_equal(o[t], v[kr, h].numpy())) and abs(lse[t] - s_exp) <= 1e-14 * max(1, abs(s_exp))
                    ok0 &= bool(np.all(dq[t] == 0))
                else:
                    ok0 &= bool(np.isneginf(lse[t]) and np.all(o[t] == 0))
    res.append(("window_zero_width_diagonal", ok0))
    # one visible key per row: dk = 0 and dv_j = dO of the row that sees key j
    dv_exp = np.zeros_like(dv)
    for b in range(len(lq)):
        for ii in range(lq[b]):
            jj = ii + lk[b] - lq[b]
            if 0 <= jj < lk[b]:
                for h in range(H):
                    dv_exp[(ck[b] + jj) * H + h] += do[cq[b] + ii, h].numpy()
    res.append(("window_zero_width_grads", bool(np.all(dk == 0) and np.allclose(dv, dv_exp, rtol=0, atol=1e-15))))
    # band of the diagonal key and the one before it (window (1, 0)), Sq = Sk segment:
    # a two-term softmax, o = (e_a v_{i-1} + e_b v_i) / (e_a + e_b)
    o, lse, *_ = run(window=(1, 0))
    ok2 = True
    b = 0
    for ii in range(1, lq[b]):
        r = cq[b] + ii
        for h in range(H):
            sa = sc * float(torch.dot(q[r, h], k[ck[b] + ii - 1, h]))
            sb = sc * float(torch.dot(q[r, h], k[ck[b] + ii, h]))
            mx = max(sa, sb)
            ea, eb = math.exp(sa - mx), math.exp(sb - mx)
            o_exp = (ea * v[ck[b] + ii - 1, h].numpy() + eb * v[ck[b] + ii, h].numpy()) / (ea + eb)
            ok2 &= bool(np.allclose(o[r * H + h], o_exp, rtol=1e-13, atol=1e-14))
            ok2 &= abs(lse[r * H + h] - (mx + math.log(ea + eb))) <= 1e-13
    res.append(("window_two_key_band", ok2))
    # same band, right side: window (0, 1) on the Sq < Sk segment sees keys ii+d and ii+d+1
    o, lse, *_ = run(window=(0, 1))
    ok3 = True
    b = 1
    d = lk[b] - lq[b]
    for ii in range(lq[b]):
        r = cq[b] + ii
        j0, j1 = ii + d, min(ii + d + 1, lk[b] - 1)
        for h in range(H):
            ss = [sc * float(torch.dot(q[r, h], k[ck[b] + j, h])) for j in range(j0, j1 + 1)]
            mx = max(ss)
            es = [math.exp(x - mx) for x in ss]
            o_exp = sum(e * v[ck[b] + j, h].numpy() for e, j in zip(es, range(j0, j1 + 1))) / sum(es)
            ok3 &= bool(np.allclose(o[r * H + h], o_exp, rtol=1e-13, atol=1e-14))
    res.append(("window_right_band", ok3))
    # windows wider than every segment: identical to no mask; (-1, 0): identical to causal
    full = run()
    wide = run(window=(64, 64))
    res.append(("window_wide_is_unmasked", all(np.array_equal(a, b_) for a, b_ in zip(full, wide))))
    cz = run(causal=True)
    wc = run(window=(-1, 0))
    res.append(("window_left_unbounded_is_causal", all(np.array_equal(a, b_) for a, b_ in zip(cz, wc))))
    # gradients of a general band against masked torch autograd
    wl, wr = 2, 1
    o, lse, dq, dk, dv = run(window=(wl, wr))
    ro, rl, rdq, rdk, rdv = _torch_masked_reference(
        q, k, v, do, cq, ck, sc,
        lambda i, j, d: (j >= i + d - wl) & (j <= i + d + wr))
    res.append(("window_out", np.allclose(o, ro.reshape(-1, D).numpy(), rtol=1e-12, atol=1e-13)))
    res.append(("window_lse", np.allclose(lse, rl.reshape(-1).numpy(), rtol=1e-12, atol=1e-13)))
    res.append(("window_dq", np.allclose(dq, rdq.reshape(-1, D).numpy(), rtol=1e-10, atol=1e-12)))
    res.append(("window_dk", np.allclose(dk, rdk.reshape(-1, D).numpy(), rtol=1e-10, atol=1e-12)))
    res.append(("window_dv", np.allclose(dv, rdv.reshape(-1, D).numpy(), rtol=1e-10, atol=1e-12)))
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
            with np.errstate(divide="ignore", invalid="ignore"):  # a planted mistake may zero P[ii, 0]
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
    res += _window_checks(lib, seed)
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
    g = json.loads(pathlib.Path(GOLDEN).read_text())
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


LEFT_EDGE = "    if (window_left >= 0 && diag - window_left > a) a = diag - window_left;"
RIGHT_EDGE = "    if (window_right >= 0 && diag + window_right + 1 < e) e = diag + window_right + 1;"

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
    ("kv segment start of the next segment", "const int64_t k0 = pb->cu_k[b];",
     "const int64_t k0 = pb->cu_k[b] + (b > 0);"),
    ("delta from dO.v instead of dO.o", "E[ii] = dot(doi, oi, D);", "E[ii] = dot(doi, doi, D);"),
    ("head stride ignored", "int64_t off = row * rs + (int64_t)h * hs;", "int64_t off = row * rs;"),
    ("causal diagonal one key early", RIGHT_EDGE, RIGHT_EDGE.replace("+ 1 < e) e = diag + window_right + 1;",
                                                                     "< e) e = diag + window_right;")),
    ("causal diagonal aligned top-left", "const int64_t diag = ii + (Sk - Sq);", "const int64_t diag = ii;"),
    ("mask missing on the key side", "if (jj < jlo || jj >= jhi) continue;", "(void)jj;"),
    ("key-side mask misses the left edge", "if (jj < jlo || jj >= jhi) continue;", "if (jj >= jhi) continue;"),
    ("window left edge one key late", LEFT_EDGE, LEFT_EDGE.replace("a = diag - window_left;",
                                                                   "a = diag - window_left + 1;")),
    ("window left side ignored", LEFT_EDGE, LEFT_EDGE.replace("if (window_left >= 0 &&", "if (0 &&")),
    ("window right width ignored", RIGHT_EDGE, RIGHT_EDGE.replace("window_right + 1", "1")),
    ("window sides swapped", LEFT_EDGE + "\n" + RIGHT_EDGE,
     LEFT_EDGE.replace("window_left", "window_right") + "\n" + RIGHT_EDGE.replace("window_right", "window_left")),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = pathlib.Path(oracle._SRC).read_text()
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
