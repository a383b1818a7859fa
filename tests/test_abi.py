"""The C ABI on the host (no GPU needed): the library builds and loads, it
exports every entry point include/sa.h declares, argument checks return their
error codes before anything touches a device, and the product package never
reaches the oracle."""
import ctypes
import os
import re

import pytest

from indexer_selected_sparse_score_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_symbols():
    names = []
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if hdr.endswith(".h"):
            text = open(os.path.join(ROOT, "include", hdr)).read()
            names += re.findall(r"SA_API\s+[\w\s\*]+?\b(sa_\w+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert "sa_fused_decode" in names and len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert set(binding.EXPORTED) <= set(names)


def _ia(**kw):
    base = dict(B=2, T=3, H_I=16, D_I=64, N_c=100, r=2, q_seq=16, q_pos=16, q_I=16, q_dtype=0,
                q_scale=None, w=16, k_I=16, k_dtype=1, k_scale=16, k_seq_stride=0)
    base.update(kw)
    return binding.IndexArgs(*[base[f] for f, _ in binding.IndexArgs._fields_])


def _aa(**kw):
    base = dict(H=16, D=128, W=8, R=8, Q=16, Kw=16, Vw=16, Kc=16, Vc=16, sink=None, scale=0.088,
                w_seq_stride=0, c_seq_stride=0)
    base.update(kw)
    return binding.AttnArgs(*[base[f] for f, _ in binding.AttnArgs._fields_])


def _call_fused(lib, ia, aa, K=8, ws=256, ws_bytes=1 << 20, out=256):
    return lib.sa_fused_decode(ctypes.byref(ia) if ia is not None else None,
                               ctypes.byref(aa) if aa is not None else None, K, None, out, ws,
                               ws_bytes, None)


def test_workspace_size(lib):
    n = lib.sa_workspace_size(ctypes.byref(_ia()), ctypes.byref(_aa()), 8)
    assert n > 256 and n % 256 == 0
    assert lib.sa_workspace_size(ctypes.byref(_ia(B=0)), None, 8) == 0
    assert lib.sa_workspace_size(ctypes.byref(_ia()), None, -1) == 0


@pytest.mark.parametrize("ia,aa,K,status", [
    (None, _aa(), 8, binding.SA_ERR_INVALID_ARG),
    (_ia(T=-1), _aa(), 8, binding.SA_ERR_INVALID_ARG),
    (_ia(r=0), _aa(), 8, binding.SA_ERR_INVALID_ARG),
    (_ia(D_I=96), _aa(), 8, binding.SA_ERR_UNSUPPORTED),
    (_ia(H_I=129), _aa(), 8, binding.SA_ERR_UNSUPPORTED),
    (_ia(q_dtype=7), _aa(), 8, binding.SA_ERR_INVALID_ARG),
    (_ia(k_I=24), _aa(), 8, binding.SA_ERR_INVALID_ARG),        # misaligned
    (_ia(), _aa(H=24), 8, binding.SA_ERR_UNSUPPORTED),
    (_ia(), _aa(D=64), 8, binding.SA_ERR_UNSUPPORTED),
    (_ia(), _aa(R=4), 8, binding.SA_ERR_INVALID_ARG),           # R < W
    (_ia(), _aa(scale=float("nan")), 8, binding.SA_ERR_INVALID_ARG),
    (_ia(), _aa(Q=None), 8, binding.SA_ERR_INVALID_ARG),
    (_ia(), _aa(), -1, binding.SA_ERR_INVALID_ARG),
])
def test_fused_rejects_bad_arguments(lib, ia, aa, K, status):
    assert _call_fused(lib, ia, aa, K) == status
    assert lib.sa_last_error_detail()


def test_workspace_checks(lib):
    assert _call_fused(lib, _ia(), _aa(), ws=None) == binding.SA_ERR_WORKSPACE
    assert _call_fused(lib, _ia(), _aa(), ws_bytes=300) == binding.SA_ERR_WORKSPACE
    assert _call_fused(lib, _ia(), _aa(), ws=264) == binding.SA_ERR_INVALID_ARG


def test_status_strings(lib):
    for s in range(7):
        assert lib.sa_status_string(s)


def test_product_package_never_reaches_the_oracle():
    pkg = os.path.join(ROOT, "indexer_selected_sparse_score_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "oracle.h" not in text and "liboracle" not in text, f


def test_candidate_words(lib):
    assert lib.sa_candidate_words(32768, 8) == 128
    assert lib.sa_candidate_words(20, 4) == 1
    assert lib.sa_candidate_words(257, 8) == 2       # 33 blocks
    assert lib.sa_candidate_words(100, 1000) == 1    # one short block
    assert lib.sa_candidate_words(0, 8) == 0
    assert lib.sa_candidate_words(100, 0) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(block_size=0), binding.SA_ERR_INVALID_ARG),
    (dict(topk_blocks=-1), binding.SA_ERR_INVALID_ARG),
    (dict(ia=_ia(N_c=32768 * 8 + 1)), binding.SA_ERR_UNSUPPORTED),   # 32769 blocks
    (dict(ia=_ia(N_c=(1 << 30) + 1), block_size=1 << 20), binding.SA_ERR_UNSUPPORTED),  # row too long
    (dict(scores=None), binding.SA_ERR_INVALID_ARG),
    (dict(cand=None), binding.SA_ERR_INVALID_ARG),
    (dict(cand=258), binding.SA_ERR_INVALID_ARG),                     # misaligned
    (dict(ws=None), binding.SA_ERR_WORKSPACE),
    (dict(ws_bytes=64), binding.SA_ERR_WORKSPACE),
    (dict(ia=_ia(r=0)), binding.SA_ERR_INVALID_ARG),
    (dict(ld=99), binding.SA_ERR_INVALID_ARG),                        # score rows shorter than N_c
])
def test_candidate_blocks_rejects_bad_arguments(lib, kw, status):
    a = dict(scores=256, ld=None, ia=_ia(), block_size=8, topk_blocks=4, cand=256, ws=256, ws_bytes=256)
    a.update(kw)
    ld = a["ia"].N_c if a["ld"] is None else a["ld"]
    st = lib.sa_candidate_blocks(a["scores"], ld, ctypes.byref(a["ia"]), a["block_size"], a["topk_blocks"],
                                 a["cand"], a["ws"], a["ws_bytes"], None)
    assert st == status
    assert lib.sa_last_error_detail()


@pytest.mark.parametrize("kw,status", [
    (dict(block_size=0), binding.SA_ERR_INVALID_ARG),
    (dict(K=-1), binding.SA_ERR_INVALID_ARG),
    (dict(cand=None), binding.SA_ERR_INVALID_ARG),
    (dict(idx=None), binding.SA_ERR_INVALID_ARG),
    (dict(cand=258), binding.SA_ERR_INVALID_ARG),
    (dict(ws=None), binding.SA_ERR_WORKSPACE),
    (dict(ia=_ia(N_c=(1 << 30) + 1)), binding.SA_ERR_UNSUPPORTED),
    (dict(ld=50), binding.SA_ERR_INVALID_ARG),
])
def test_topk_candidates_rejects_bad_arguments(lib, kw, status):
    a = dict(scores=256, ld=None, ia=_ia(), K=8, cand=256, block_size=8, idx=256, ws=256, ws_bytes=256)
    a.update(kw)
    ld = a["ia"].N_c if a["ld"] is None else a["ld"]
    st = lib.sa_topk_candidates(a["scores"], ld, ctypes.byref(a["ia"]), a["K"], a["cand"], a["block_size"],
                                a["idx"], a["ws"], a["ws_bytes"], None)
    assert st == status


def test_candidate_calls_with_no_tokens_enqueue_nothing(lib):
    # T = 0: valid arguments and nothing to do (no device is touched)
    ia = _ia(T=0, q_seq=None, q_pos=None)
    assert lib.sa_candidate_blocks(None, 100, ctypes.byref(ia), 8, 4, None, 256, 256, None) == binding.SA_OK
    assert lib.sa_topk_candidates(None, 100, ctypes.byref(ia), 8, None, 8, None, 256, 256, None) == binding.SA_OK


@pytest.mark.parametrize("kw,status", [
    (dict(ia=_ia(k_seq_stride=100 * 64 - 64)), binding.SA_ERR_INVALID_ARG),    # below N_c * D_I
    (dict(ia=_ia(k_seq_stride=100 * 64 + 32)), binding.SA_ERR_INVALID_ARG),    # not whole rows
    (dict(aa=_aa(w_seq_stride=7 * 128)), binding.SA_ERR_INVALID_ARG),         # below R * D
    (dict(aa=_aa(w_seq_stride=8 * 128 + 8)), binding.SA_ERR_INVALID_ARG),
    (dict(aa=_aa(c_seq_stride=99 * 128)), binding.SA_ERR_INVALID_ARG),        # below N_c * D
    (dict(aa=_aa(c_seq_stride=100 * 128 + 64)), binding.SA_ERR_INVALID_ARG),
    (dict(aa=_aa(c_seq_stride=(1 << 31) * 128)), binding.SA_ERR_UNSUPPORTED),  # rows past 31 bits
])
def test_sequence_strides_are_checked(lib, kw, status):
    a = dict(ia=_ia(), aa=_aa())
    a.update(kw)
    assert _call_fused(lib, a["ia"], a["aa"]) == status
    assert lib.sa_last_error_detail()
    assert lib.sa_workspace_size(ctypes.byref(a["ia"]), ctypes.byref(a["aa"]), 8) == 0


def test_padded_strides_are_accepted(lib):
    # a cache with room for 4 x more rows per sequence than are in use
    n = lib.sa_workspace_size(ctypes.byref(_ia(k_seq_stride=400 * 64)),
                              ctypes.byref(_aa(w_seq_stride=32 * 128, c_seq_stride=400 * 128)), 8)
    assert n == lib.sa_workspace_size(ctypes.byref(_ia()), ctypes.byref(_aa()), 8)


def test_score_row_stride_is_checked(lib):
    ia = _ia()
    assert lib.sa_topk(256, 99, ctypes.byref(ia), 8, 256, 256, 256, None) == binding.SA_ERR_INVALID_ARG
    assert lib.sa_indexer_scores(ctypes.byref(ia), 256, 64, 256, 1 << 20, None) == binding.SA_ERR_INVALID_ARG
    ia0 = _ia(T=0, q_seq=None, q_pos=None)
    assert lib.sa_topk(None, 128, ctypes.byref(ia0), 8, None, 256, 256, None) == binding.SA_OK


def test_attention_head_dims(lib):
    # dim 512 (the released V4.1 shape) with up to 64 heads; 128 heads of dim 512 do not fit
    assert lib.sa_workspace_size(ctypes.byref(_ia()), ctypes.byref(_aa(H=64, D=512)), 8) > 0
    assert lib.sa_workspace_size(ctypes.byref(_ia()), ctypes.byref(_aa(H=16, D=512)), 8) > 0
    assert _call_fused(lib, _ia(), _aa(H=128, D=512)) == binding.SA_ERR_UNSUPPORTED
    assert _call_fused(lib, _ia(), _aa(H=64, D=256)) == binding.SA_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw,status", [
    (dict(rows=-1), binding.SA_ERR_INVALID_ARG),
    (dict(dim=64), binding.SA_ERR_UNSUPPORTED),
    (dict(x=None), binding.SA_ERR_INVALID_ARG),
    (dict(x=264), binding.SA_ERR_INVALID_ARG),          # not 16-byte aligned
    (dict(codes=258), binding.SA_ERR_INVALID_ARG),
    (dict(dst=256, dst_rows=-1), binding.SA_ERR_INVALID_ARG),
    (dict(ws=None), binding.SA_ERR_WORKSPACE),
])
def test_rotate_quant_rejects_bad_arguments(lib, kw, status):
    a = dict(x=256, rows=4, dim=128, dst=None, dst_rows=0, codes=256, scales=256, ws=256, ws_bytes=256)
    a.update(kw)
    st = lib.sa_rotate_quant(a["x"], a["rows"], a["dim"], a["dst"], a["dst_rows"], a["codes"], a["scales"],
                             a["ws"], a["ws_bytes"], None)
    assert st == status


def test_rotate_quant_with_no_rows_enqueues_nothing(lib):
    assert lib.sa_rotate_quant(None, 0, 128, None, 0, None, None, 256, 256, None) == binding.SA_OK


@pytest.mark.parametrize("kw,status", [
    (dict(r=1), binding.SA_ERR_INVALID_ARG),
    (dict(D=48), binding.SA_ERR_UNSUPPORTED),
    (dict(D=2048), binding.SA_ERR_UNSUPPORTED),
    (dict(B=70000), binding.SA_ERR_INVALID_ARG),
    (dict(eps=float("nan")), binding.SA_ERR_INVALID_ARG),
    (dict(kv=None), binding.SA_ERR_INVALID_ARG),
    (dict(out=258), binding.SA_ERR_INVALID_ARG),
])
def test_compress_prefill_rejects_bad_arguments(lib, kw, status):
    a = dict(kv=256, score=256, B=2, S=8, D=64, r=4, weight=256, eps=1e-6, out=256, kvs=None, scs=None)
    a.update(kw)
    st = lib.sa_compress_prefill(a["kv"], a["score"], a["B"], a["S"], a["D"], a["r"], a["weight"], a["eps"], a["out"],
                                 a["kvs"], a["scs"], None)
    assert st == status


def test_compress_prefill_states_go_together(lib):
    assert lib.sa_compress_prefill(256, 256, 2, 9, 64, 4, 256, 1e-6, 256, 256, None, None) == binding.SA_ERR_INVALID_ARG


def test_compress_prefill_with_no_group_enqueues_nothing(lib):
    assert lib.sa_compress_prefill(None, None, 2, 3, 64, 4, None, 1e-6, None, None, None, None) == binding.SA_OK


@pytest.mark.parametrize("kw,status", [
    (dict(r=1), binding.SA_ERR_INVALID_ARG),
    (dict(D=40), binding.SA_ERR_UNSUPPORTED),
    (dict(pos=None), binding.SA_ERR_INVALID_ARG),
    (dict(kvs=258), binding.SA_ERR_INVALID_ARG),
    (dict(ws=None), binding.SA_ERR_WORKSPACE),
])
def test_compress_decode_rejects_bad_arguments(lib, kw, status):
    a = dict(kv=256, score=256, pos=256, B=2, D=64, r=4, kvs=256, scs=256, weight=256, eps=1e-6, out=256, ws=256,
             ws_bytes=256)
    a.update(kw)
    st = lib.sa_compress_decode(a["kv"], a["score"], a["pos"], a["B"], a["D"], a["r"], a["kvs"], a["scs"],
                                a["weight"], a["eps"], a["out"], a["ws"], a["ws_bytes"], None)
    assert st == status


def _rope(**kw):
    base = dict(dim=64, base=160000.0, factor=16.0, original_seq_len=65536, beta_fast=32.0, beta_slow=1.0)
    base.update(kw)
    return binding.RopeArgs(*[base[f] for f, _ in binding.RopeArgs._fields_])


@pytest.mark.parametrize("kw,status", [
    (dict(D_I=64), binding.SA_ERR_UNSUPPORTED),
    (dict(rope=_rope(dim=66)), binding.SA_ERR_INVALID_ARG),
    (dict(rope=_rope(dim=132)), binding.SA_ERR_INVALID_ARG),
    (dict(rope=_rope(base=1.0)), binding.SA_ERR_INVALID_ARG),
    (dict(rope=None), binding.SA_ERR_INVALID_ARG),
    (dict(stride=100 * 128 - 128), binding.SA_ERR_INVALID_ARG),
    (dict(kproj=264), binding.SA_ERR_INVALID_ARG),
    (dict(seq=None), binding.SA_ERR_INVALID_ARG),
    (dict(ws=None), binding.SA_ERR_WORKSPACE),
    (dict(n=-1), binding.SA_ERR_INVALID_ARG),
])
def test_index_key_publish_rejects_bad_arguments(lib, kw, status):
    a = dict(kproj=256, n=4, D_I=128, seq=256, grp=256, r=4, weight=256, eps=1e-6, rope=_rope(), k_I=256,
             k_scale=256, B=2, N_rows=100, stride=0, ws=256, ws_bytes=256)
    a.update(kw)
    st = lib.sa_index_key_publish(a["kproj"], a["n"], a["D_I"], a["seq"], a["grp"], a["r"], a["weight"], a["eps"],
                                  ctypes.byref(a["rope"]) if a["rope"] is not None else None, a["k_I"], a["k_scale"],
                                  a["B"], a["N_rows"], a["stride"], a["ws"], a["ws_bytes"], None)
    assert st == status


def test_wait_budget_argument_check():
    """sa_set_wait_budget touches no device: a negative bound is refused, 0 restores the default."""
    lib = binding.load()
    assert lib.sa_set_wait_budget(-5) == binding.SA_ERR_INVALID_ARG
    assert lib.sa_set_wait_budget(1000) == binding.SA_OK
    assert lib.sa_set_wait_budget(0) == binding.SA_OK
