"""The seeded workloads at full size, in the launch configuration the
benchmark times, checked against the oracle on EVERY output row: every
(sequence, query head) of the decode workloads and every (query, head) of the
prefill workloads.  At these sizes the kernels take paths that small cases
barely reach (balanced tile ranges with fix-up slots, runs that start inside a
split, the longest-first order of chunked prefill), so nothing is sampled."""
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


def _compare(out, lse, ref, ref_lse, int8, what):
    o = out.float().cpu().numpy().reshape(ref.shape)
    l = lse.cpu().numpy().reshape(-1)
    assert_close(o, ref, int8=int8, what=what)
    assert_lse_close(l, ref_lse, what=what)


@pytest.mark.parametrize("name", ["tiny_decode", "paged_gqa_decode", "int8_long_decode", "ring_window_decode",
                                  "paged_decode_f32io"])
def test_decode_workload(name):
    g = si.make_workload(name, device="cuda")
    lse = torch.empty((g.batch, g.n_heads), dtype=torch.float32, device="cuda")
    out = attn.decode(g, lse_out=lse, out_f32=bool(si.WORKLOADS[name].get("out_f32")))
    torch.cuda.synchronize()
    cpu = g.to("cpu")
    del g
    ref, ref_lse = oracle.decode(cpu)
    _compare(out, lse, ref, ref_lse, cpu.int8, name)


def test_tiered_workload():
    g = si.make_workload("tiered_int8_decode", device="cuda")
    lse = torch.empty((g.batch, g.n_heads), dtype=torch.float32, device="cuda")
    out = attn.decode_tiered(g, lse_out=lse)
    torch.cuda.synchronize()
    cpu = g.to("cpu")
    del g
    ref, ref_lse = oracle.decode_tiered(cpu)
    _compare(out, lse, ref, ref_lse, True, "tiered_int8_decode")


@pytest.mark.parametrize("name", ["vision_2304", "swa_softcap_prefill"])
def test_prefill_workload(name):
    g = si.make_workload(name, device="cuda")
    lse = torch.empty((g.seq_len, g.n_heads), dtype=torch.float32, device="cuda")
    out = attn.prefill(g, lse_out=lse)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.prefill(g.to("cpu"))
    _compare(out, lse, ref, ref_lse, False, name)


def test_chunked_prefill_workload():
    g = si.make_workload("chunked_prefill_paged", device="cuda")
    lse = torch.empty((g.total_q, g.n_heads), dtype=torch.float32, device="cuda")
    out = attn.prefill_paged(g, lse_out=lse)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.prefill_paged(g.to("cpu"))
    _compare(out, lse, ref, ref_lse, False, "chunked_prefill_paged")
