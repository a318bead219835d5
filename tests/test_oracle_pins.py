"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: the pages'
own parameter arithmetic (tests/golden), closed forms, special cases that
reduce to a library routine, mask enumeration by interval reasoning, brute
force with scipy's softmax on the full score matrix, and layout equivalences.
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    return rows


def _decode_case_from_arrays(q, k, v, lens, scale, window=0, softcap=0.0):
    """Contiguous f16 decode case from float arrays (rounded to f16)."""
    q = torch.tensor(np.asarray(q), dtype=torch.float16)
    k = torch.tensor(np.asarray(k), dtype=torch.float16)
    v = torch.tensor(np.asarray(v), dtype=torch.float16)
    B, Hq, D = q.shape
    return si.DecodeCase(q=q, k=k, v=v, kv_len=torch.tensor(lens, dtype=torch.int32),
                         batch=B, n_heads=Hq, n_kv_heads=k.shape[2], head_dim=D,
                         cap=k.shape[1], window=window, softcap=softcap, scale=scale,
                         lens=list(lens))


def _prefill_case_from_arrays(q, k, v, causal, scale, window=0, softcap=0.0):
    q = torch.tensor(np.asarray(q), dtype=torch.float16)
    k = torch.tensor(np.asarray(k), dtype=torch.float16)
    v = torch.tensor(np.asarray(v), dtype=torch.float16)
    S, Hq, D = q.shape
    return si.PrefillCase(q=q, k=k, v=v, seq_len=S, n_heads=Hq, n_kv_heads=k.shape[1],
                          head_dim=D, causal=causal, window=window, softcap=softcap,
                          scale=scale)


# ---------------------------------------------------------------- brute force
def _kept_set(pos, L, causal, window):
    """Kept key positions, built as an interval (not via the oracle's predicate)."""
    if causal:
        lo = 0 if window <= 0 else max(0, pos - window + 1)
        hi = min(L - 1, pos)
    else:
        lo = 0 if window <= 0 else max(0, pos - window + 1)
        hi = L - 1 if window <= 0 else min(L - 1, pos + window - 1)
    return set(range(lo, hi + 1))


def _brute(qrows, K, V, positions, L, causal, window, softcap, scale, dtype=np.float64):
    """Full score matrix + scipy softmax; qrows [n, D], K/V [L, D]."""
    qrows = qrows.astype(dtype)
    K = K.astype(dtype)
    V = V.astype(dtype)
    S = (qrows @ K.T) * dtype(scale)
    if softcap > 0:
        S = dtype(softcap) * np.tanh(S / dtype(softcap))
    mask = np.full(S.shape, False)
    for r, pos in enumerate(positions):
        for j in _kept_set(pos, L, causal, window):
            mask[r, j] = True
    Sm = np.where(mask, S, -np.inf).astype(np.float64)
    P = scipy.special.softmax(Sm, axis=1)
    O = P @ V.astype(np.float64)
    lse = scipy.special.logsumexp(Sm, axis=1)
    return O, lse, P


# ---------------------------------------------------------------- pins
def test_f16_decoder_matches_numpy_for_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_powers_of_two_worked_example():
    (o0, o1, lse_ref), = _golden_rows("powers_of_two_example.txt")
    q = [[[1.0, 0.0]]]
    k = [[[[0.0, 0.0]], [[1.0, 0.0]], [[2.0, 0.0]]]]
    v = [[[[1.0, 0.0]], [[0.0, 1.0]], [[1.0, 1.0]]]]
    case = _decode_case_from_arrays(q, k, v, [3], scale=math.log(2.0))
    out, lse = oracle.decode(case)
    assert out[0, 0] == pytest.approx(o0, abs=1e-15)
    assert out[0, 1] == pytest.approx(o1, abs=1e-15)
    assert lse[0] == pytest.approx(lse_ref, abs=1e-15)


def test_scale_rule_golden():
    # the library takes the scale as an argument; the pages' rule for it
    for scalar, head_dim, want in _golden_rows("scale_from_query_pre_attn_scalar.txt"):
        got = 1.0 / math.sqrt(scalar) if scalar else 1.0 / math.sqrt(head_dim)
        assert got == want


@pytest.mark.parametrize("D", [4, 64])
def test_single_key_returns_its_value_row(D):
    rng = np.random.default_rng(0)
    q = rng.standard_normal((1, 2, D))
    k = rng.standard_normal((1, 5, 1, D))
    v = rng.standard_normal((1, 5, 1, D))
    case = _decode_case_from_arrays(q, k, v, [1], scale=0.3)
    out, lse = oracle.decode(case)
    v0 = case.v[0, 0, 0].double().numpy()
    assert np.array_equal(out[0], v0) and np.array_equal(out[1], v0)
    # prefill row 0 under a causal mask also sees exactly one key
    pc = _prefill_case_from_arrays(rng.standard_normal((3, 1, D)), rng.standard_normal((3, 1, D)),
                                   rng.standard_normal((3, 1, D)), causal=True, scale=0.7)
    o, _ = oracle.prefill(pc, rows=[(0, 0)])
    assert np.array_equal(o[0], pc.v[0, 0].double().numpy())


def test_constant_values_return_that_value():
    rng = np.random.default_rng(1)
    D, L = 16, 37
    vbar = rng.standard_normal(D)
    q = rng.standard_normal((2, 4, D))
    k = rng.standard_normal((2, L, 2, D))
    v = np.broadcast_to(vbar, (2, L, 2, D))
    case = _decode_case_from_arrays(q, k, v, [L, 11], scale=0.25, softcap=3.0, window=7)
    out, _ = oracle.decode(case)
    vb = case.v[0, 0, 0].double().numpy()
    assert np.allclose(out, vb[None, :], rtol=0, atol=1e-14)


def test_zero_scale_gives_mean_of_visible_rows():
    rng = np.random.default_rng(2)
    S, D, W = 9, 8, 4
    pc = _prefill_case_from_arrays(rng.standard_normal((S, 2, D)), rng.standard_normal((S, 1, D)),
                                   rng.standard_normal((S, 1, D)), causal=True, scale=0.0,
                                   window=W)
    out, lse = oracle.prefill(pc)
    V = pc.v[:, 0].double().numpy()
    for i in range(S):
        lo = max(0, i - W + 1)
        want = V[lo:i + 1].mean(axis=0)
        assert np.allclose(out[i * 2], want, atol=1e-15, rtol=0)
        assert np.allclose(out[i * 2 + 1], want, atol=1e-15, rtol=0)
        assert lse[i * 2] == pytest.approx(math.log(i + 1 - lo), abs=1e-15)


def _one_hot_prefill(S, causal, window, softcap=0.0, seed=3):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((S, 1, S))
    k = rng.standard_normal((S, 1, S))
    v = np.eye(S)[:, None, :]            # v_j = e_j  => output row = weights
    return _prefill_case_from_arrays(q, k, v, causal=causal, scale=0.2, window=window,
                                     softcap=softcap)


@pytest.mark.parametrize("causal,window", [(True, 0), (True, 1), (True, 3), (False, 0),
                                           (False, 2), (False, 5)])
def test_mask_enumeration_and_weights_sum_to_one(causal, window):
    S = 12
    pc = _one_hot_prefill(S, causal, window)
    W, _ = oracle.prefill(pc)
    for i in range(S):
        kept = {j for j in range(S) if W[i, j] != 0.0}
        assert kept == _kept_set(i, S, causal, window)
        assert np.all(W[i] >= 0)
        assert W[i].sum() == pytest.approx(1.0, abs=1e-14)


def test_causal_window_pair_count():
    # causal row i keeps i+1 keys; with a window, min(i+1, W)
    S, Wn = 16, 5
    pc = _one_hot_prefill(S, True, Wn)
    W, _ = oracle.prefill(pc)
    counts = (W != 0).sum(axis=1)
    assert list(counts) == [min(i + 1, Wn) for i in range(S)]


def test_decode_window_clamp_golden():
    for total, window, kv_start, kept_len in _golden_rows("window_clamp.txt"):
        total, window, kv_start, kept_len = int(total), int(window), int(kv_start), int(kept_len)
        D = max(total, 2)
        rng = np.random.default_rng(total * 100 + window)
        q = rng.standard_normal((1, 1, D))
        k = rng.standard_normal((1, total, 1, D))
        v = np.eye(D)[:total][None, :, None, :]
        case = _decode_case_from_arrays(q, k, v, [total], scale=0.1, window=window)
        out, _ = oracle.decode(case)
        kept = [j for j in range(total) if out[0, j] != 0.0]
        assert kept == list(range(kv_start, kv_start + kept_len))


def test_softcap_saturation_closed_form():
    # c = 1 and logits of +-1000: tanh saturates to +-1 in double, so the two
    # weights are 1 : e^2 regardless of the raw logits.
    D = 2
    q = [[[1.0, 0.0]]]
    k = [[[[-1000.0, 0.0]], [[1000.0, 0.0]]]]
    v = [[[[1.0, 0.0]], [[0.0, 1.0]]]]
    case = _decode_case_from_arrays(q, k, v, [2], scale=1.0, softcap=1.0)
    out, lse = oracle.decode(case)
    e2 = math.exp(2.0)
    assert out[0, 0] == pytest.approx(1.0 / (1.0 + e2), abs=1e-15)
    assert out[0, 1] == pytest.approx(e2 / (1.0 + e2), abs=1e-15)
    assert lse[0] == pytest.approx(1.0 + math.log(1.0 + math.exp(-2.0)), abs=1e-14)
    # without the cap the large logit wins outright
    nocap = _decode_case_from_arrays(q, k, v, [2], scale=1.0, softcap=0.0)
    o2, _ = oracle.decode(nocap)
    assert o2[0, 0] == 0.0 and o2[0, 1] == 1.0


def test_huge_softcap_equals_no_cap():
    case = si.make_decode_case(2, 4, 2, 16, [9, 30], seed=7)
    a, la = oracle.decode(case)
    case.softcap = 1e12
    b, lb = oracle.decode(case)
    assert np.allclose(a, b, atol=1e-12, rtol=0) and np.allclose(la, lb, atol=1e-12)


@pytest.mark.parametrize("S,Hq,Hkv,D,causal,window,softcap", [
    (1, 1, 1, 4, True, 0, 0.0),
    (5, 4, 2, 8, True, 0, 0.0),
    (17, 6, 3, 16, True, 3, 2.5),
    (17, 4, 1, 16, False, 0, 0.0),
    (13, 2, 2, 8, False, 4, 1.5),
    (33, 8, 2, 32, True, 8, 0.0),
])
def test_prefill_matches_brute_force(S, Hq, Hkv, D, causal, window, softcap):
    pc = si.make_prefill_case(S, Hq, Hkv, D, seed=S * 10 + Hq, causal=causal, window=window,
                              softcap=softcap, scale=0.37)
    out, lse = oracle.prefill(pc)
    q = pc.q.double().numpy()
    K = np.repeat(pc.k.double().numpy(), Hq // Hkv, axis=1)    # explicit repeat-KV
    V = np.repeat(pc.v.double().numpy(), Hq // Hkv, axis=1)
    for h in range(Hq):
        for dt in (np.float64, np.longdouble):
            O, L, _ = _brute(q[:, h], K[:, h], V[:, h], list(range(S)), S, causal, window,
                             softcap, 0.37, dtype=dt)
            assert np.allclose(out[h::Hq], O, atol=1e-12, rtol=0)
            assert np.allclose(lse[h::Hq], L, atol=1e-12, rtol=0)


def _dequant_contiguous(case):
    """Float64 K/V [B, cap, Hkv, D] from a contiguous case (int8: codes * scales)."""
    if case.int8:
        ks = case.k_scales.double().numpy().transpose(0, 2, 1)[..., None]   # [B, cap, Hkv, 1]
        vs = case.v_scales.double().numpy().transpose(0, 2, 1)[..., None]
        return case.k.numpy().astype(np.float64) * ks, case.v.numpy().astype(np.float64) * vs
    return case.k.double().numpy(), case.v.double().numpy()


@pytest.mark.parametrize("int8", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,D,lens,window,softcap", [
    (1, 4, 2, 64, [128], 0, 0.0),
    (3, 8, 2, 16, [1, 17, 40], 0, 0.0),
    (2, 6, 3, 8, [25, 9], 6, 0.0),
    (2, 4, 4, 32, [50, 33], 0, 4.0),
])
def test_decode_matches_brute_force(int8, B, Hq, Hkv, D, lens, window, softcap):
    case = si.make_decode_case(B, Hq, Hkv, D, lens, seed=B * 31 + D, int8=int8,
                               window=window, softcap=softcap, scale=0.21)
    out, lse = oracle.decode(case)
    K, V = _dequant_contiguous(case)
    q = case.q.double().numpy()
    G = Hq // Hkv
    for b in range(B):
        L = lens[b]
        for h in range(Hq):
            O, LS, _ = _brute(q[b, h][None], K[b, :L, h // G], V[b, :L, h // G], [L - 1], L,
                              True, window, softcap, 0.21)
            assert np.allclose(out[b * Hq + h], O[0], atol=1e-12, rtol=0)
            assert lse[b * Hq + h] == pytest.approx(LS[0], abs=1e-12)


@pytest.mark.parametrize("int8", [False, True])
@pytest.mark.parametrize("page_size", [1, 8, 16])
def test_paged_layout_equals_contiguous_exactly(int8, page_size):
    case = si.make_decode_case(3, 4, 2, 16, [5, 33, 20], seed=11, int8=int8, cap=40)
    paged = si.paged_from_contiguous(case, page_size, seed=12)
    a, la = oracle.decode(case)
    b, lb = oracle.decode(paged)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_seeded_paged_case_matches_brute_force():
    case = si.make_decode_case(4, 4, 2, 16, (3, 60), seed=13, page_size=8, int8=True)
    out, _ = oracle.decode(case)
    pt = case.page_table.numpy()
    kc, vc = case.k.numpy().astype(np.float64), case.v.numpy().astype(np.float64)
    ks, vs = case.k_scales.double().numpy(), case.v_scales.double().numpy()
    q = case.q.double().numpy()
    for b, L in enumerate(case.lens):
        rows = [(pt[b, t // 8], t % 8) for t in range(L)]
        for h in range(4):
            g = h // 2
            K = np.stack([kc[p, r, g] * ks[p, g, r] for p, r in rows])
            V = np.stack([vc[p, r, g] * vs[p, g, r] for p, r in rows])
            O, _, _ = _brute(q[b, h][None], K, V, [L - 1], L, True, 0, 0.0, case.scale)
            assert np.allclose(out[b * 4 + h], O[0], atol=1e-12, rtol=0)


def test_gqa_mapping_contiguous_groups():
    # permuting kv heads, with the query-head groups permuted alongside,
    # permutes the outputs the same way (mapping g = h // G)
    case = si.make_decode_case(2, 6, 3, 8, [7, 12], seed=17)
    out, _ = oracle.decode(case)
    perm = [2, 0, 1]
    G = 2
    qperm = [perm[h // G] * G + h % G for h in range(6)]
    pcase = si.make_decode_case(2, 6, 3, 8, [7, 12], seed=17)
    pcase.k = case.k[:, :, perm].contiguous()
    pcase.v = case.v[:, :, perm].contiguous()
    pcase.q = case.q[:, qperm].contiguous()
    pout, _ = oracle.decode(pcase)
    out = out.reshape(2, 6, 8)
    pout = pout.reshape(2, 6, 8)
    assert np.array_equal(pout, out[:, qperm])
    # G = 1 is plain multi-head attention: head h reads kv head h
    mha = si.make_decode_case(1, 3, 3, 8, [9], seed=18)
    o, _ = oracle.decode(mha)
    K, V = mha.k.double().numpy(), mha.v.double().numpy()
    for h in range(3):
        O, _, _ = _brute(mha.q[0, h].double().numpy()[None], K[0, :9, h], V[0, :9, h], [8], 9,
                         True, 0, 0.0, mha.scale)
        assert np.allclose(o[h], O[0], atol=1e-12)


def test_zero_length_sequence_gives_zeros():
    case = si.make_decode_case(2, 2, 1, 8, [0, 4], seed=19, cap=8)
    out, lse = oracle.decode(case)
    assert np.all(out[:2] == 0) and np.all(np.isneginf(lse[:2]))
    assert np.all(np.isfinite(out[2:]))


def test_row_selection_matches_full_run():
    pc = si.make_prefill_case(20, 4, 2, 16, seed=21, causal=True, window=6, softcap=5.0)
    full, fl = oracle.prefill(pc)
    rows = [(0, 0), (19, 3), (7, 2), (13, 1)]
    part, pl = oracle.prefill(pc, rows=rows)
    for n, (i, h) in enumerate(rows):
        assert np.array_equal(part[n], full[i * 4 + h]) and pl[n] == fl[i * 4 + h]
    case = si.make_decode_case(3, 4, 2, 16, [5, 9, 2], seed=22)
    full, fl = oracle.decode(case)
    part, pl = oracle.decode(case, rows=[(2, 3), (0, 1)])
    assert np.array_equal(part[0], full[2 * 4 + 3]) and np.array_equal(part[1], full[1])


def test_int8_encoding_rule():
    # the generator's encoding: s = f16(max|x|/127), codes in [-127, 127],
    # |x - code*s| <= s/2 (plus the f16 rounding of s), zero rows -> zero codes
    x = si.f16_normal((64, 32), seed=23)
    x[5] = 0
    codes, scales = si.quantize_int8_rows(x)
    xf, sf, cf = x.double(), scales.double(), codes.double()
    assert codes.abs().max() <= 127
    assert torch.all(cf[5] == 0) and sf[5] == 0
    err = (xf - cf * sf[:, None]).abs().max(dim=1).values
    assert torch.all(err <= sf * 0.5 * (1 + 1e-3) + 1e-12)


# ---- chunked prefill / multi-token decode over a paged cache -----------------

def _chunk_from_prefill(pc, page_size, seed):
    """A one-sequence chunk holding all of a prefill case's tokens (ctx 0), with
    its K/V scattered into a paged pool by a seeded permutation."""
    S, Hkv, D, P = pc.seq_len, pc.n_kv_heads, pc.head_dim, page_size
    max_pages = (S + P - 1) // P
    n_pages = max_pages + 2
    perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(seed))
    pt = perm[:max_pages].view(1, max_pages).to(torch.int32)
    kp = torch.zeros((n_pages, P, Hkv, D), dtype=torch.float16)
    vp = torch.zeros((n_pages, P, Hkv, D), dtype=torch.float16)
    for i in range(max_pages):
        t0, t1 = i * P, min((i + 1) * P, S)
        kp[int(pt[0, i]), :t1 - t0] = pc.k[t0:t1]
        vp[int(pt[0, i]), :t1 - t0] = pc.v[t0:t1]
    return si.ChunkCase(q=pc.q, k=kp, v=vp, q_start=torch.tensor([0, S], dtype=torch.int32),
                        kv_len=torch.tensor([S], dtype=torch.int32), page_table=pt, batch=1,
                        n_heads=pc.n_heads, n_kv_heads=Hkv, head_dim=D, page_size=P,
                        max_pages=max_pages, max_q=S, window=pc.window, softcap=pc.softcap,
                        scale=pc.scale, q_lens=[S], kv_lens=[S])


@pytest.mark.parametrize("page_size", [1, 8, 16])
@pytest.mark.parametrize("window", [0, 9])
def test_whole_sequence_chunk_equals_causal_prefill(page_size, window):
    # a chunk with no prior context is causal prefill of the same tokens: the
    # page gather and the query positions must reproduce the contiguous path
    pc = si.make_prefill_case(37, 4, 2, 32, seed=5, causal=True, window=window, softcap=3.0, scale=0.3)
    cc = _chunk_from_prefill(pc, page_size, seed=7)
    a, la = oracle.prefill(pc)
    b, lb = oracle.prefill_paged(cc)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_one_token_chunks_equal_decode():
    # decode is the one-new-token case: the query sits at kv_len - 1
    cc = si.make_chunked_case(3, 4, 2, 32, [1, 1, 1], [40, 0, 17], seed=11, page_size=8, window=10)
    dc = si.DecodeCase(q=cc.q, k=cc.k, v=cc.v, kv_len=cc.kv_len, batch=3, n_heads=4, n_kv_heads=2,
                       head_dim=32, cap=cc.max_pages * cc.page_size, page_table=cc.page_table,
                       page_size=cc.page_size, max_pages=cc.max_pages, window=10, scale=cc.scale)
    a, la = oracle.prefill_paged(cc)
    b, lb = oracle.decode(dc)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


@pytest.mark.parametrize("window,softcap", [(0, 0.0), (6, 0.0), (0, 2.5)])
def test_chunked_matches_brute_force(window, softcap):
    # scipy softmax over the full score matrix with an independently built mask
    cc = si.make_chunked_case(3, 4, 2, 16, [5, 1, 9], [11, 0, 20], seed=13, page_size=4,
                              window=window, softcap=softcap, scale=0.4)
    got, lse = oracle.prefill_paged(cc)
    q = cc.q.double().numpy()
    k, v, pt = cc.k.double().numpy(), cc.v.double().numpy(), cc.page_table.numpy()
    P, G = cc.page_size, cc.n_heads // cc.n_kv_heads
    row = 0
    for b in range(cc.batch):
        L, n = cc.kv_lens[b], cc.q_lens[b]
        keys = np.stack([k[pt[b, t // P], t % P] for t in range(L)])     # [L, Hkv, D]
        vals = np.stack([v[pt[b, t // P], t % P] for t in range(L)])
        for i in range(n):
            pos = L - n + i
            for h in range(cc.n_heads):
                s = cc.scale * keys[:, h // G, :] @ q[row + i, h]
                if softcap > 0:
                    s = softcap * np.tanh(s / softcap)
                t = np.arange(L)
                keep = t <= pos
                if window > 0:
                    keep &= (pos - t) < window
                s = np.where(keep, s, -np.inf)
                p = scipy.special.softmax(s)
                r = (row + i) * cc.n_heads + h
                np.testing.assert_allclose(got[r], p @ vals[:, h // G, :], rtol=0, atol=1e-12)
                np.testing.assert_allclose(lse[r], scipy.special.logsumexp(s), rtol=0, atol=1e-12)
        row += n


def test_chunk_longer_than_its_cache_sees_nothing_before_position_zero():
    # kv_len < q_len: the first q_len - kv_len queries sit at negative positions
    cc = si.make_chunked_case(1, 2, 1, 16, [6], [0], seed=17, page_size=4)
    cc.kv_len = torch.tensor([4], dtype=torch.int32)     # only 4 of the 6 tokens are cached
    got, lse = oracle.prefill_paged(cc)
    got, lse = got.reshape(6, 2, 16), lse.reshape(6, 2)
    assert np.all(got[:2] == 0) and np.all(np.isneginf(lse[:2]))
    # query 2 sits at position 0 and sees key 0 only: its value row
    v0 = cc.v[int(cc.page_table[0, 0]), 0, 0].double().numpy()
    np.testing.assert_allclose(got[2, 0], v0, rtol=0, atol=1e-12)


def test_empty_chunks_are_skipped():
    cc = si.make_chunked_case(3, 2, 2, 16, [0, 3, 0], [10, 5, 0], seed=19, page_size=4)
    got, _ = oracle.prefill_paged(cc)
    assert got.shape == (3 * 2, 16)
    ref, _ = oracle.prefill_paged(si.make_chunked_case(3, 2, 2, 16, [0, 3, 0], [10, 5, 0], seed=19,
                                                       page_size=4), rows=[(r, h) for r in range(3)
                                                                          for h in range(2)])
    assert np.array_equal(got, ref)


# ---- ring (sliding-window) cache ---------------------------------------------

@pytest.mark.parametrize("int8", [False, True])
@pytest.mark.parametrize("ring,window", [(16, 0), (32, 0), (32, 20), (48, 100)])
def test_ring_equals_contiguous_with_its_window(int8, ring, window):
    # a ring of R slots keeps the last min(L, R, W) logical tokens: the same as a
    # contiguous cache of every token with the window min(W, R)
    lens = [5, 16, 47, 100]
    cc = si.make_decode_case(4, 4, 2, 32, lens, seed=41, int8=int8, cap=104, window=window)
    rc = si.ring_from_contiguous(cc, ring)
    w_eff = ring if window <= 0 else min(window, ring)
    cc.window = w_eff
    a, la = oracle.decode(cc)
    b, lb = oracle.decode(rc)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_ring_matches_brute_force():
    cc = si.make_decode_case(2, 2, 1, 16, [70, 9], seed=43, cap=72)
    rc = si.ring_from_contiguous(cc, 32)
    got, lse = oracle.decode(rc)
    q = cc.q.double().numpy()
    for b, L in enumerate([70, 9]):
        keep = min(L, 32)
        ts = list(range(L - keep, L))
        K = np.stack([rc.k[b, t % 32, 0].double().numpy() for t in ts])
        V = np.stack([rc.v[b, t % 32, 0].double().numpy() for t in ts])
        for h in range(2):
            s = rc.scale * K @ q[b, h]
            p = scipy.special.softmax(s)
            np.testing.assert_allclose(got[b * 2 + h], p @ V, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[b * 2 + h], scipy.special.logsumexp(s), rtol=0, atol=1e-12)


# ---- tiered (cold cache + hot ring) decode -----------------------------------

def _tiered_brute(c, b, h):
    """Tiered decode of one (sequence, head) straight from the definition: cold
    token j at position j, hot token i at cold_len + i in ring slot
    (hot_start + i) mod ring, the ring holding the newest hot_ring hot tokens,
    the window by position from the query (the newest token); scipy softmax."""
    G = c.n_heads // c.n_kv_heads
    g = h // G
    cap = c.max_pages * c.page_size if c.page_table is not None else c.cap
    Lc = min(max(int(c.kv_len[b]), 0), cap)
    Lh = max(int(c.hot_len[b]), 0)
    qpos = Lc + Lh - 1
    keys, vals = [], []

    def cold_row(t, which):
        cache = c.k if which == 0 else c.v
        scales = c.k_scales if which == 0 else c.v_scales
        if c.page_table is not None:
            page, r = int(c.page_table[b, t // c.page_size]), t % c.page_size
            x = cache[page, r, g].double().numpy()
            sc = float(scales[page, g, r]) if c.int8 else 1.0
        else:
            x = cache[b, t, g].double().numpy()
            sc = float(scales[b, g, t]) if c.int8 else 1.0
        return x * sc

    for j in range(Lc):
        if c.window > 0 and qpos - j >= c.window:
            continue
        keys.append(cold_row(j, 0))
        vals.append(cold_row(j, 1))
    for i in range(max(0, Lh - c.hot_ring), Lh):
        if c.window > 0 and qpos - (Lc + i) >= c.window:
            continue
        slot = (int(c.hot_start[b]) + i) % c.hot_ring
        keys.append(c.hot_k[b, slot, g].double().numpy())
        vals.append(c.hot_v[b, slot, g].double().numpy())
    if not keys:
        return np.zeros(c.head_dim), -math.inf
    K, V = np.stack(keys), np.stack(vals)
    s = c.scale * (K @ c.q[b, h].double().numpy())
    if c.softcap > 0:
        s = c.softcap * np.tanh(s / c.softcap)
    return scipy.special.softmax(s) @ V, scipy.special.logsumexp(s)


@pytest.mark.parametrize("int8,page_size", [(False, 0), (True, 0), (False, 8), (True, 16)])
@pytest.mark.parametrize("window,softcap", [(0, 0.0), (7, 0.0), (30, 20.0)])
def test_tiered_matches_brute_force(int8, page_size, window, softcap):
    # ragged cold and hot lengths: an empty sequence, a hot tier that has
    # overwritten its ring (40 > 16), rings starting mid-way, windows that end
    # inside the hot tier, inside the cold tier, or not at all
    c = si.make_tiered_case(4, 4, 2, 16, [0, 25, 3, 50], [0, 5, 40, 16], 16, seed=61 + page_size,
                            hot_starts=[0, 13, 7, 15], int8=int8, page_size=page_size, window=window,
                            softcap=softcap)
    got, lse = oracle.decode_tiered(c)
    for b in range(4):
        for h in range(4):
            o, l = _tiered_brute(c, b, h)
            np.testing.assert_allclose(got[b * 4 + h], o, rtol=0, atol=1e-12)
            if math.isinf(l):
                assert lse[b * 4 + h] == -math.inf
            else:
                np.testing.assert_allclose(lse[b * 4 + h], l, rtol=0, atol=1e-12)


@pytest.mark.parametrize("int8", [False, True])
@pytest.mark.parametrize("window", [0, 12])
def test_tiered_with_no_hot_tokens_is_decode_over_the_cold_cache(int8, window):
    c = si.make_tiered_case(3, 4, 2, 16, [1, 40, 77], [0, 0, 0], 32, seed=63, int8=int8, page_size=16,
                            window=window)
    cold = si.DecodeCase(**{k: v for k, v in c.__dict__.items() if k in si.DecodeCase.__dataclass_fields__})
    a, la = oracle.decode_tiered(c)
    b, lb = oracle.decode(cold)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


@pytest.mark.parametrize("window", [0, 9, 30])
def test_tiered_equals_one_contiguous_cache_of_both_tiers(window):
    # hot tokens all still in the ring: cold tokens then hot tokens in one
    # contiguous cache, decoded with the same window, is the same attention
    c = si.make_tiered_case(3, 4, 2, 16, [0, 20, 33], [6, 0, 16], 16, seed=65, hot_starts=[3, 9, 15],
                            window=window)
    lens = [int(c.kv_len[b]) + int(c.hot_len[b]) for b in range(3)]
    k = torch.zeros((3, 64, 2, 16), dtype=torch.float16)
    v = torch.zeros_like(k)
    for b in range(3):
        Lc = int(c.kv_len[b])
        k[b, :Lc], v[b, :Lc] = c.k[b, :Lc], c.v[b, :Lc]
        for i in range(int(c.hot_len[b])):
            slot = (int(c.hot_start[b]) + i) % 16
            k[b, Lc + i], v[b, Lc + i] = c.hot_k[b, slot], c.hot_v[b, slot]
    flat = si.DecodeCase(q=c.q, k=k, v=v, kv_len=torch.tensor(lens, dtype=torch.int32), batch=3, n_heads=4,
                         n_kv_heads=2, head_dim=16, cap=64, window=window, scale=c.scale, lens=lens)
    a, la = oracle.decode_tiered(c)
    b, lb = oracle.decode(flat)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)
    np.testing.assert_allclose(la, lb, rtol=0, atol=1e-13)


# ---- f32 queries --------------------------------------------------------------

def test_f32_queries_that_are_f16_values_match_the_f16_path():
    # a binary32 query holding exactly the f16 values is the same query
    c = si.make_decode_case(3, 4, 2, 32, [1, 40, 77], seed=71, int8=True, page_size=16, window=30)
    c32 = si.DecodeCase(**{**c.__dict__, "q": c.q.float()})
    a, la = oracle.decode(c)
    b, lb = oracle.decode(c32)
    assert np.array_equal(a, b) and np.array_equal(la, lb)
    t = si.make_tiered_case(2, 4, 2, 16, [10, 30], [5, 40], 16, seed=72)
    t32 = si.TieredCase(**{**t.__dict__, "q": t.q.float()})
    a, la = oracle.decode_tiered(t)
    b, lb = oracle.decode_tiered(t32)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_f32_queries_match_brute_force():
    c = si.make_decode_case(2, 4, 2, 16, [9, 33], seed=73, q_f32=True, softcap=10.0)
    assert c.q.dtype == torch.float32 and not torch.equal(c.q, c.q.half().float())
    got, lse = oracle.decode(c)
    for b, L in enumerate([9, 33]):
        K = c.k[b, :L].double().numpy()
        V = c.v[b, :L].double().numpy()
        for h in range(4):
            s = c.scale * (K[:, h // 2] @ c.q[b, h].double().numpy())
            s = 10.0 * np.tanh(s / 10.0)
            p = scipy.special.softmax(s)
            np.testing.assert_allclose(got[b * 4 + h], p @ V[:, h // 2], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[b * 4 + h], scipy.special.logsumexp(s), rtol=0, atol=1e-12)
