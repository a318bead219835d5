"""C-ABI checks that need no GPU: the library builds and loads, exports every
entry point include/attn.h declares, plans workspaces, and rejects bad
arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

import attention_split_kv_gb300 as attn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    attn.build()
    return attn.load()


def _declared_entry_points():
    src = open(os.path.join(ROOT, "include", "attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_0-9]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert sorted(attn.exported_symbols) == _declared_entry_points()


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_entry_points():
        assert hasattr(lib, name), name
    assert attn.attn_version().startswith("libattn")


def test_library_has_no_driver_link_dependency():
    # the runtime is linked statically and the driver is reached through the
    # runtime's entry-point query, so the library loads on a machine without one
    out = os.popen("ldd %s" % attn.lib_path()).read()
    assert "libcuda.so" not in out and "libcudart.so" not in out


def test_workspace_plan(lib):
    # B=32, Hq=32, Hkv=8, D=128, max_kv 8192: G=4 -> one head group per kv head
    n = attn.attn_decode_workspace_size(32, 32, 8, 128, 8192)
    assert n > 0
    # explicit split: items <= B*Hkv*(ceil(8192/512)+1); lse + o per item and head
    n512 = attn.attn_decode_workspace_size(32, 32, 8, 128, 8192, 512)
    items = 32 * 8 * (8192 // 512 + 1)
    assert n512 >= items * 4 * (128 + 1) * 4
    assert attn.attn_decode_workspace_size(32, 30, 8, 128, 8192) == 0    # Hq % Hkv
    assert attn.attn_decode_workspace_size(32, 32, 8, 96, 8192) == 0     # head_dim
    assert attn.attn_decode_workspace_size(32, 32, 8, 128, 8192, 24) == 0  # split not % 16
    assert attn.attn_decode_workspace_size(5000, 32, 8, 128, 8192) == 0  # batch limit


FAKE = 1 << 20   # a non-null, 16-byte aligned address never dereferenced on the host


def _decode(**kw):
    args = dict(q=FAKE, k_cache=FAKE, v_cache=FAKE, kv_len=FAKE, page_table=None, page_size=0,
                max_pages_per_seq=0, n_pages=0, max_kv=128, k_scales=None, v_scales=None,
                kv_dtype=attn.ATTN_KV_F16, batch=1, n_heads=4, n_kv_heads=2, head_dim=64, window=0,
                softcap=0.0, scale=0.125, split_keys=0, out=FAKE, lse_out=None, workspace=FAKE,
                workspace_bytes=1 << 30, stream=0)
    args.update(kw)
    return attn.load().attn_decode(*[args[k] for k in (
        "q", "k_cache", "v_cache", "kv_len", "page_table", "page_size", "max_pages_per_seq", "n_pages",
        "max_kv", "k_scales", "v_scales", "kv_dtype", "batch", "n_heads", "n_kv_heads", "head_dim",
        "window", "softcap", "scale", "split_keys", "out", "lse_out", "workspace", "workspace_bytes",
        "stream")])


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), attn.ATTN_EINVAL),
    (dict(n_heads=5), attn.ATTN_EINVAL),
    (dict(head_dim=96), attn.ATTN_EUNSUPPORTED),
    (dict(window=-1), attn.ATTN_EINVAL),
    (dict(softcap=-1.0), attn.ATTN_EINVAL),
    (dict(softcap=float("inf")), attn.ATTN_EINVAL),
    (dict(scale=float("nan")), attn.ATTN_EINVAL),
    (dict(kv_dtype=7), attn.ATTN_EINVAL),
    (dict(kv_dtype=attn.ATTN_KV_INT8), attn.ATTN_EINVAL),                 # scales missing
    (dict(kv_dtype=attn.ATTN_KV_INT8, k_scales=FAKE, v_scales=FAKE, max_kv=100), attn.ATTN_EUNSUPPORTED),
    (dict(page_table=FAKE, page_size=12, max_pages_per_seq=8, n_pages=8), attn.ATTN_EUNSUPPORTED),
    (dict(page_table=FAKE, page_size=4, max_pages_per_seq=8, n_pages=8, kv_dtype=attn.ATTN_KV_INT8,
          k_scales=FAKE, v_scales=FAKE), attn.ATTN_EUNSUPPORTED),
    (dict(page_table=FAKE, page_size=16, max_pages_per_seq=0, n_pages=8), attn.ATTN_EINVAL),
    (dict(split_keys=24), attn.ATTN_EINVAL),
    (dict(workspace_bytes=16), attn.ATTN_EINVAL),
    (dict(workspace=None), attn.ATTN_EINVAL),
    (dict(q=FAKE + 2), attn.ATTN_EINVAL),                                  # misaligned
    (dict(batch=5000), attn.ATTN_EUNSUPPORTED),
    (dict(max_kv=0), attn.ATTN_EINVAL),
])
def test_decode_rejects_bad_arguments_on_host(lib, kw, status):
    assert _decode(**kw) == status
    assert attn.attn_last_error()


def _decode_ring(**kw):
    args = dict(q=FAKE, k_ring=FAKE, v_ring=FAKE, seq_len=FAKE, ring_size=64, k_scales=None, v_scales=None,
                kv_dtype=attn.ATTN_KV_F16, batch=1, n_heads=4, n_kv_heads=2, head_dim=64, window=0,
                softcap=0.0, scale=0.125, split_keys=0, out=FAKE, lse_out=None, workspace=FAKE,
                workspace_bytes=1 << 30, stream=0)
    args.update(kw)
    return attn.load().attn_decode_ring(*[args[k] for k in (
        "q", "k_ring", "v_ring", "seq_len", "ring_size", "k_scales", "v_scales", "kv_dtype", "batch",
        "n_heads", "n_kv_heads", "head_dim", "window", "softcap", "scale", "split_keys", "out", "lse_out",
        "workspace", "workspace_bytes", "stream")])


@pytest.mark.parametrize("kw,status", [
    (dict(ring_size=0), attn.ATTN_EUNSUPPORTED),
    (dict(ring_size=40), attn.ATTN_EUNSUPPORTED),        # not a multiple of 16
    (dict(ring_size=-32), attn.ATTN_EUNSUPPORTED),
    (dict(seq_len=None), attn.ATTN_EINVAL),
    (dict(head_dim=96), attn.ATTN_EUNSUPPORTED),
    (dict(kv_dtype=attn.ATTN_KV_INT8), attn.ATTN_EINVAL),  # scales missing
    (dict(window=-1), attn.ATTN_EINVAL),
    (dict(workspace_bytes=16), attn.ATTN_EINVAL),
])
def test_decode_ring_rejects_bad_arguments_on_host(lib, kw, status):
    assert _decode_ring(**kw) == status
    assert attn.attn_last_error()


def _decode_tiered(**kw):
    args = dict(q=FAKE, q_dtype=attn.ATTN_F16, out_dtype=attn.ATTN_F16, cold_k=FAKE, cold_v=FAKE,
                cold_k_scales=None, cold_v_scales=None,
                cold_dtype=attn.ATTN_KV_F16, cold_len=FAKE, cold_page_table=None, cold_page_size=0,
                cold_max_pages_per_seq=0, cold_n_pages=0, cold_max_kv=128, hot_k=FAKE, hot_v=FAKE, hot_len=FAKE,
                hot_start=FAKE, hot_ring=64, batch=1, n_heads=4, n_kv_heads=2, head_dim=64, window=0, softcap=0.0,
                scale=0.125, split_keys=0, out=FAKE, lse_out=None, workspace=FAKE, workspace_bytes=1 << 30,
                stream=0)
    args.update(kw)
    return attn.load().attn_decode_tiered(*[args[k] for k in (
        "q", "q_dtype", "cold_k", "cold_v", "cold_k_scales", "cold_v_scales", "cold_dtype", "cold_len",
        "cold_page_table", "cold_page_size", "cold_max_pages_per_seq", "cold_n_pages", "cold_max_kv", "hot_k", "hot_v",
        "hot_len", "hot_start", "hot_ring", "batch", "n_heads", "n_kv_heads", "head_dim", "window", "softcap", "scale",
        "split_keys", "out", "out_dtype", "lse_out", "workspace", "workspace_bytes", "stream")])


@pytest.mark.parametrize("kw,status", [
    (dict(hot_ring=0), attn.ATTN_EUNSUPPORTED),
    (dict(hot_ring=24), attn.ATTN_EUNSUPPORTED),
    (dict(hot_start=None), attn.ATTN_EINVAL),
    (dict(hot_k=None), attn.ATTN_EINVAL),
    (dict(cold_len=None), attn.ATTN_EINVAL),
    (dict(cold_dtype=attn.ATTN_KV_INT8), attn.ATTN_EINVAL),            # cold scales missing
    (dict(cold_page_table=FAKE, cold_page_size=12, cold_max_pages_per_seq=4, cold_n_pages=4),
     attn.ATTN_EUNSUPPORTED),
    (dict(head_dim=80), attn.ATTN_EUNSUPPORTED),
    (dict(workspace_bytes=64), attn.ATTN_EINVAL),
    (dict(hot_v=FAKE + 4), attn.ATTN_EINVAL),                            # misaligned
    (dict(q_dtype=2), attn.ATTN_EINVAL),
    (dict(out_dtype=7), attn.ATTN_EINVAL),
])
def test_decode_tiered_rejects_bad_arguments_on_host(lib, kw, status):
    assert _decode_tiered(**kw) == status
    assert attn.attn_last_error()


def test_tiered_workspace_is_both_plans(lib):
    a = attn.attn_decode_workspace_size(4, 32, 8, 128, 8192)
    h = attn.attn_decode_workspace_size(4, 32, 8, 128, 1024)
    t = attn.attn_decode_tiered_workspace_size(4, 32, 8, 128, 8192, 1024)
    assert t >= a + h and t < a + h + 256
    assert attn.attn_decode_tiered_workspace_size(4, 32, 8, 128, 8192, 1000) == 0    # ring % 16


def _decode_ex(**kw):
    args = dict(q=FAKE, q_dtype=attn.ATTN_F32, k_cache=FAKE, v_cache=FAKE, kv_len=FAKE, page_table=None,
                page_size=0, max_pages_per_seq=0, n_pages=0, max_kv=128, ring_size=0, k_scales=None, v_scales=None,
                kv_dtype=attn.ATTN_KV_F16, batch=1, n_heads=4, n_kv_heads=2, head_dim=64, window=0, softcap=0.0,
                scale=0.125, split_keys=0, out=FAKE, out_dtype=attn.ATTN_F32, lse_out=None, workspace=FAKE,
                workspace_bytes=1 << 30, stream=0)
    args.update(kw)
    return attn.load().attn_decode_ex(*[args[k] for k in (
        "q", "q_dtype", "k_cache", "v_cache", "kv_len", "page_table", "page_size", "max_pages_per_seq", "n_pages",
        "max_kv", "ring_size", "k_scales", "v_scales", "kv_dtype", "batch", "n_heads", "n_kv_heads", "head_dim",
        "window", "softcap", "scale", "split_keys", "out", "out_dtype", "lse_out", "workspace", "workspace_bytes",
        "stream")])


@pytest.mark.parametrize("kw,status", [
    (dict(q_dtype=3), attn.ATTN_EINVAL),
    (dict(out_dtype=-1), attn.ATTN_EINVAL),
    (dict(ring_size=20), attn.ATTN_EUNSUPPORTED),
    (dict(ring_size=32, page_table=FAKE, page_size=16, max_pages_per_seq=2, n_pages=4), attn.ATTN_EINVAL),
    (dict(q=FAKE + 8), attn.ATTN_EINVAL),                                 # misaligned
    (dict(head_dim=32), attn.ATTN_EUNSUPPORTED),
    (dict(workspace_bytes=16), attn.ATTN_EINVAL),
])
def test_decode_ex_rejects_bad_arguments_on_host(lib, kw, status):
    assert _decode_ex(**kw) == status
    assert attn.attn_last_error()


def _prefill(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, seq_len=128, n_heads=4, n_kv_heads=2, head_dim=64, causal=1,
                window=0, softcap=0.0, scale=0.125, out=FAKE, lse_out=None, stream=0)
    args.update(kw)
    return attn.load().attn_prefill(*[args[k] for k in (
        "q", "k", "v", "seq_len", "n_heads", "n_kv_heads", "head_dim", "causal", "window", "softcap",
        "scale", "out", "lse_out", "stream")])


@pytest.mark.parametrize("kw,status", [
    (dict(k=None), attn.ATTN_EINVAL),
    (dict(n_heads=3), attn.ATTN_EINVAL),
    (dict(head_dim=80), attn.ATTN_EUNSUPPORTED),
    (dict(window=-3), attn.ATTN_EINVAL),
    (dict(softcap=-0.5), attn.ATTN_EINVAL),
    (dict(seq_len=-1), attn.ATTN_EINVAL),
    (dict(out=FAKE + 8), attn.ATTN_EINVAL),
    (dict(seq_len=0), attn.ATTN_OK),          # nothing to do, nothing launched
])
def test_prefill_rejects_bad_arguments_on_host(lib, kw, status):
    assert _prefill(**kw) == status


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(attn, "_lib", None)
    monkeypatch.setattr(attn, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(attn.AttnLibraryMissing):
        attn.attn_version()


def _prefill_paged(**kw):
    args = dict(q=FAKE, k_cache=FAKE, v_cache=FAKE, q_start=FAKE, kv_len=FAKE, page_table=FAKE, page_size=16,
                max_pages=4, n_pages=8, batch=2, total_q=10, max_q=8, n_heads=4, n_kv_heads=2, head_dim=64,
                window=0, softcap=0.0, scale=0.125, out=FAKE, lse_out=None, stream=0)
    args.update(kw)
    return attn.load().attn_prefill_paged(*[args[k] for k in (
        "q", "k_cache", "v_cache", "q_start", "kv_len", "page_table", "page_size", "max_pages", "n_pages",
        "batch", "total_q", "max_q", "n_heads", "n_kv_heads", "head_dim", "window", "softcap", "scale", "out",
        "lse_out", "stream")])


@pytest.mark.parametrize("kw,status", [
    (dict(q_start=None), attn.ATTN_EINVAL),
    (dict(page_table=None), attn.ATTN_EINVAL),
    (dict(batch=0), attn.ATTN_EINVAL),
    (dict(total_q=-1), attn.ATTN_EINVAL),
    (dict(n_heads=5), attn.ATTN_EINVAL),
    (dict(head_dim=80), attn.ATTN_EUNSUPPORTED),
    (dict(page_size=12), attn.ATTN_EUNSUPPORTED),
    (dict(page_size=4), attn.ATTN_EUNSUPPORTED),
    (dict(n_pages=0), attn.ATTN_EINVAL),
    (dict(window=-2), attn.ATTN_EINVAL),
    (dict(softcap=float("nan")), attn.ATTN_EINVAL),
    (dict(scale=float("inf")), attn.ATTN_EINVAL),
    (dict(out=FAKE + 2), attn.ATTN_EINVAL),
])
def test_prefill_paged_rejects_bad_arguments_on_the_host(lib, kw, status):
    assert _prefill_paged(**kw) == status
    assert "attn_prefill_paged" in attn.attn_last_error()


def test_prefill_paged_with_no_queries_is_a_no_op(lib):
    assert _prefill_paged(total_q=0) == attn.ATTN_OK
    assert _prefill_paged(max_q=0) == attn.ATTN_OK
