"""GPU parity of attn_prefill_paged (chunked prefill / multi-token decode over a
paged cache) against the oracle, through the C ABI: several tiles, ragged
chunks, empty chunks, chunks longer than their cache, page sizes below and above
the key tile, and the bit-identity with contiguous causal prefill."""
import numpy as np
import pytest
import torch

import attention_split_kv_gb300 as attn
import oracle
import seeded_inputs as si
from parity_util import assert_close, assert_lse_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    attn.build()
    attn.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield
    assert attn.attn_device_status() == attn.ATTN_OK


def _run(case):
    g = case.to("cuda")
    lse = torch.empty((max(case.total_q, 1), case.n_heads), dtype=torch.float32, device="cuda")
    out = torch.zeros_like(g.q)
    attn.prefill_paged(g, out=out, lse_out=lse)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()[:case.total_q], lse.cpu().numpy()[:case.total_q]


def _check(case, what):
    ref, ref_lse = oracle.prefill_paged(case)
    got, lse = _run(case)
    assert_close(got.reshape(ref.shape), ref, what=what)
    assert_lse_close(lse.reshape(-1), ref_lse, what=what)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("page_size", [8, 16, 256])
def test_chunks(D, page_size):
    # ragged chunks over several key and query tiles, one empty chunk, one decode step
    case = si.make_chunked_case(4, 4, 2, D, [130, 0, 1, 37], [300, 50, 777, 0], seed=D + page_size,
                                page_size=page_size)
    _check(case, "D=%d P=%d" % (D, page_size))


@pytest.mark.parametrize("n_seq", [5, 40])
def test_many_sequences_both_launch_orders(n_seq):
    # up to 128 (sequence, query tile) pairs are ranked longest first inside the
    # kernel; more pairs take the plain (tile, head, sequence) grid.  40 sequences
    # of up to 4 query tiles give 160 pairs.
    rng = np.random.default_rng(n_seq)
    q_lens = [int(x) for x in rng.integers(0, 200, n_seq)]
    ctx = [int(x) for x in rng.integers(0, 500, n_seq)]
    q_lens[0] = 500   # the longest chunk sets the grid: 4 query tiles
    case = si.make_chunked_case(n_seq, 4, 2, 128, q_lens, ctx, seed=90 + n_seq, page_size=16)
    _check(case, "%d sequences" % n_seq)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 2), (6, 2)])
def test_chunks_gqa(Hq, Hkv):
    case = si.make_chunked_case(2, Hq, Hkv, 128, [64, 200], [500, 129], seed=Hq * 10 + Hkv, page_size=16)
    _check(case, "GQA %d/%d" % (Hq, Hkv))


@pytest.mark.parametrize("window,softcap", [(1, 0.0), (50, 0.0), (300, 5.0), (0, 30.0)])
def test_chunks_window_softcap(window, softcap):
    case = si.make_chunked_case(3, 8, 2, 128, [90, 1, 260], [400, 99, 1000], seed=window + 3, page_size=32,
                                window=window, softcap=softcap, scale=1.0 / 16.0)
    _check(case, "window %d softcap %g" % (window, softcap))


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("page_size", [16, 128])
def test_whole_sequence_chunk_is_bit_identical_to_causal_prefill(D, page_size):
    # no prior context: the paged kernel must produce the contiguous kernel's bits
    S = 300
    pc = si.make_prefill_case(S, 4, 2, D, seed=D + 1, causal=True, window=0)
    P = page_size
    max_pages = (S + P - 1) // P
    n_pages = max_pages + 3
    perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(D))
    pt = perm[:max_pages].view(1, max_pages).to(torch.int32)
    kp = torch.zeros((n_pages, P, 2, D), dtype=torch.float16)
    vp = torch.zeros((n_pages, P, 2, D), dtype=torch.float16)
    for i in range(max_pages):
        t0, t1 = i * P, min((i + 1) * P, S)
        kp[int(pt[0, i]), :t1 - t0] = pc.k[t0:t1]
        vp[int(pt[0, i]), :t1 - t0] = pc.v[t0:t1]
    cc = si.ChunkCase(q=pc.q, k=kp, v=vp, q_start=torch.tensor([0, S], dtype=torch.int32),
                      kv_len=torch.tensor([S], dtype=torch.int32), page_table=pt, batch=1, n_heads=4,
                      n_kv_heads=2, head_dim=D, page_size=P, max_pages=max_pages, max_q=S, scale=pc.scale,
                      q_lens=[S], kv_lens=[S])
    a, la = _run(cc)
    g = pc.to("cuda")
    lse = torch.empty((S, 4), dtype=torch.float32, device="cuda")
    b = attn.prefill(g, lse_out=lse)
    torch.cuda.synchronize()
    assert np.array_equal(a, b.float().cpu().numpy()) and np.array_equal(la, lse.cpu().numpy())


def test_one_token_chunks_agree_with_decode():
    cc = si.make_chunked_case(3, 8, 2, 128, [1, 1, 1], [400, 0, 1300], seed=23, page_size=16)
    a, la = _run(cc)
    dc = si.DecodeCase(q=cc.q, k=cc.k, v=cc.v, kv_len=cc.kv_len, batch=3, n_heads=8, n_kv_heads=2,
                       head_dim=128, cap=cc.max_pages * 16, page_table=cc.page_table, page_size=16,
                       max_pages=cc.max_pages, scale=cc.scale).to("cuda")
    lse = torch.empty((3, 8), dtype=torch.float32, device="cuda")
    b = attn.decode(dc, lse_out=lse)
    torch.cuda.synchronize()
    assert np.abs(a.reshape(3, 8, 128) - b.float().cpu().numpy()).max() <= 2e-3
    assert np.abs(la.reshape(3, 8) - lse.cpu().numpy()).max() <= 2e-3


def test_chunk_longer_than_its_cache():
    # kv_len < q_len: queries at negative positions keep no key (zeros, lse -inf)
    cc = si.make_chunked_case(2, 4, 2, 64, [40, 10], [0, 5], seed=29, page_size=16)
    cc.kv_len = torch.tensor([25, 15], dtype=torch.int32)
    ref, ref_lse = oracle.prefill_paged(cc)
    got, lse = _run(cc)
    assert np.all(got[:15] == 0) and np.all(np.isneginf(lse[:15]))
    assert_close(got.reshape(ref.shape), ref, what="negative positions")
    assert_lse_close(lse.reshape(-1), ref_lse, what="negative positions")


def test_invalid_page_id_is_never_read_and_is_reported():
    cc = si.make_chunked_case(2, 4, 2, 64, [20, 20], [100, 100], seed=31, page_size=16)
    cc.page_table = cc.page_table.clone()
    cc.page_table[0, 2] = 10_000_000
    got, _ = _run(cc)
    assert np.isfinite(got).all()
    assert attn.attn_device_status() == attn.ATTN_EBOUNDS
    assert attn.attn_device_status() == attn.ATTN_OK
    ref, _ = oracle.prefill_paged(cc.to("cpu"), rows=[(r, h) for r in range(20, 40) for h in range(4)])
    assert_close(got[20:40].reshape(ref.shape), ref, what="other sequence")
