"""The seeded workloads at full size, in the launch configuration the
benchmark times, checked against the oracle on sampled output rows (the
oracle computes each sampled (query, head) row exactly, one by one)."""
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


def _sample_rows(n_outer, n_heads, k, seed):
    rng = np.random.default_rng(seed)
    rows = {(0, 0), (n_outer - 1, n_heads - 1)}
    while len(rows) < k:
        rows.add((int(rng.integers(n_outer)), int(rng.integers(n_heads))))
    return sorted(rows)


@pytest.mark.parametrize("name", ["tiny_decode", "paged_gqa_decode", "int8_long_decode", "ring_window_decode",
                                  "paged_decode_f32io"])
def test_decode_workload(name):
    g = si.make_workload(name, device="cuda")
    lse = torch.empty((g.batch, g.n_heads), dtype=torch.float32, device="cuda")
    out = attn.decode(g, lse_out=lse, out_f32=bool(si.WORKLOADS[name].get("out_f32")))
    torch.cuda.synchronize()
    cpu = g.to("cpu")
    if name == "tiny_decode":
        ref, ref_lse = oracle.decode(cpu)
        assert_close(out.float().cpu().numpy().reshape(ref.shape), ref, what=name)
        assert_lse_close(lse.cpu().numpy().reshape(-1), ref_lse, what=name)
        return
    rows = _sample_rows(g.batch, g.n_heads, 24, seed=len(name))
    ref, ref_lse = oracle.decode(cpu, rows=rows)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    got = np.stack([o[b, h] for b, h in rows])
    got_lse = np.array([l[b, h] for b, h in rows])
    assert_close(got, ref, int8=g.int8, what=name)
    assert_lse_close(got_lse, ref_lse, what=name)


def test_tiered_workload():
    g = si.make_workload("tiered_int8_decode", device="cuda")
    lse = torch.empty((g.batch, g.n_heads), dtype=torch.float32, device="cuda")
    out = attn.decode_tiered(g, lse_out=lse)
    torch.cuda.synchronize()
    rows = _sample_rows(g.batch, g.n_heads, 24, seed=8)
    ref, ref_lse = oracle.decode_tiered(g.to("cpu"), rows=rows)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    assert_close(np.stack([o[b, h] for b, h in rows]), ref, int8=True, what="tiered_int8_decode")
    assert_lse_close(np.array([l[b, h] for b, h in rows]), ref_lse, what="tiered_int8_decode")


@pytest.mark.parametrize("name", ["vision_2304", "swa_softcap_prefill"])
def test_prefill_workload(name):
    g = si.make_workload(name, device="cuda")
    lse = torch.empty((g.seq_len, g.n_heads), dtype=torch.float32, device="cuda")
    out = attn.prefill(g, lse_out=lse)
    torch.cuda.synchronize()
    rows = _sample_rows(g.seq_len, g.n_heads, 64, seed=len(name))
    ref, ref_lse = oracle.prefill(g.to("cpu"), rows=rows)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    got = np.stack([o[i, h] for i, h in rows])
    got_lse = np.array([l[i, h] for i, h in rows])
    assert_close(got, ref, what=name)
    assert_lse_close(got_lse, ref_lse, what=name)


def test_chunked_prefill_workload():
    g = si.make_workload("chunked_prefill_paged", device="cuda")
    lse = torch.empty((g.total_q, g.n_heads), dtype=torch.float32, device="cuda")
    out = attn.prefill_paged(g, lse_out=lse)
    torch.cuda.synchronize()
    rows = _sample_rows(g.total_q, g.n_heads, 48, seed=6)
    ref, ref_lse = oracle.prefill_paged(g.to("cpu"), rows=rows)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    got = np.stack([o[i, h] for i, h in rows])
    got_lse = np.array([l[i, h] for i, h in rows])
    assert_close(got, ref, what="chunked_prefill_paged")
    assert_lse_close(got_lse, ref_lse, what="chunked_prefill_paged")
