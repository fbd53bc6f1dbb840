"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function include/attn.h declares, and rejects invalid
arguments before touching the device."""
import ctypes
import os
import re

import pytest
import torch

import online_softmax_fusion_gb300 as attn
from online_softmax_fusion_gb300 import build as attn_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    attn_build.build()
    return attn.lib()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_\s\*]*?\b(attn_[a-z0-9_]+)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(L):
    declared = _declared_functions()
    assert {"attn_prefill", "attn_decode_splitk", "attn_combine"} <= declared
    for name in declared:
        assert hasattr(L, name), name
    # the binding declares the same surface
    assert declared == set(attn.SIGNATURES)


def test_status_strings(L):
    for code in range(0, 9):
        s = L.attn_status_string(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert L.attn_status_string(0) == b"ok"
    assert L.attn_version() >= 100


P = ctypes.c_void_p(4096)       # aligned dummy pointer; never dereferenced
MIS = ctypes.c_void_p(4096 + 2)  # misaligned


def _prefill(L, Q=P, K=P, V=P, O=P, LSE=None, B=1, Hq=4, Hkv=2, Lq=128, Lk=128, d=128,
             causal=0, scale=0.1, slopes=None, impl=0):
    return L.attn_prefill_ex(Q, K, V, O, LSE, B, Hq, Hkv, Lq, Lk, d, causal, scale, slopes, impl,
                             None)


def test_prefill_validation_before_launch(L):
    assert _prefill(L, Q=None) == 1
    assert _prefill(L, O=None) == 1
    assert _prefill(L, B=0) == 2
    assert _prefill(L, Lq=0) == 2
    assert _prefill(L, Lk=-3) == 2
    assert _prefill(L, Hq=3, Hkv=2) == 2
    assert _prefill(L, d=96) == 3
    assert _prefill(L, d=256) == 3
    assert _prefill(L, scale=float("nan")) == 8
    assert _prefill(L, scale=float("inf")) == 8
    assert _prefill(L, K=MIS) == 7
    assert _prefill(L, LSE=ctypes.c_void_p(4098)) == 7
    assert _prefill(L, impl=7) == 3


def test_decode_validation_before_launch(L):
    def dec(Q=P, K=P, V=P, lens=None, B=2, Hq=8, Hkv=2, Lmax=1024, d=128, scale=0.1, S=0,
            Op=P, Lp=P):
        return L.attn_decode_splitk(Q, K, V, lens, B, Hq, Hkv, Lmax, d, scale, S, None, Op, Lp,
                                    None)
    assert dec(Q=None) == 1
    assert dec(Op=None) == 1
    assert dec(Hq=6, Hkv=4) == 2
    assert dec(Lmax=0) == 2
    assert dec(d=80) == 3
    assert dec(S=-1) == 4
    assert dec(scale=float("inf")) == 8
    assert dec(V=MIS) == 7
    assert L.attn_combine(None, P, 1, 1, 4, 128, P, None, None) == 1
    assert L.attn_combine(P, P, 1, 1, 0, 128, P, None, None) == 4
    assert L.attn_combine(P, P, 1, 1, 4, 32, P, None, None) == 3
    assert L.attn_combine(P, P, 0, 1, 4, 128, P, None, None) == 2


def test_valid_call_without_gpu_fails_cleanly(L):
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _prefill(L) == 5          # ATTN_ERR_CUDA, nothing launched, no crash


def test_split_geometry(L):
    # keys per split: ceil(ceil(Lk_max / S) / 64) * 64
    for Lmax, S in [(131072, 64), (32768, 16), (1000, 3), (1, 1), (65, 2), (4096, 4096)]:
        per = -(-Lmax // S)
        assert L.attn_decode_split_len(Lmax, S) == -(-per // 64) * 64
    assert L.attn_decode_split_len(0, 4) < 0
    assert L.attn_decode_split_len(100, 0) < 0
    assert L.attn_decode_num_splits(4, 8, 131072, 128, 64) == 64
    assert L.attn_decode_num_splits(1, 1, 10, 128, 64) == 10
    S = L.attn_decode_num_splits(64, 8, 32768, 128, 0)
    assert S >= 16 and (S & (S - 1)) == 0
    assert L.attn_decode_num_splits(0, 8, 32768, 128, 0) < 0
    ws = L.attn_decode_workspace_bytes(4, 64, 64, 128)
    assert ws == 4 * 64 * 64 * 128 * 4 + 4 * 64 * 64 * 4
    assert L.attn_decode_workspace_bytes(0, 64, 64, 128) == 0


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(attn, "_lib", None)
    monkeypatch.setattr(attn, "LIB_PATH", "/nonexistent/libattn.so")
    with pytest.raises(RuntimeError, match="no fallback"):
        attn.lib()


def test_binding_rejects_cpu_tensors(L):
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        attn.prefill(q, q, q)


def test_backward_validation_before_launch(L):
    def bwd(Q=P, K=P, V=P, O=P, dO=P, LSE=P, dQ=P, dK=P, dV=P, B=1, Hq=4, Hkv=2, Lq=128, Lk=128,
            d=128, causal=1, scale=0.1, ws=P, wsb=1 << 30):
        return L.attn_backward(Q, K, V, O, dO, LSE, dQ, dK, dV, B, Hq, Hkv, Lq, Lk, d, causal,
                               scale, None, ws, wsb, None)
    assert bwd(dO=None) == 1
    assert bwd(ws=None) == 1
    assert bwd(Hq=3) == 2
    assert bwd(d=96) == 3
    assert bwd(wsb=16) == 4
    assert bwd(dK=MIS) == 7
    assert L.attn_backward_workspace_bytes(2, 4, 100, 128) == 2 * 4 * 100 * 129 * 4


def test_rmsnorm_matmul_validation_before_launch(L):
    def rm(X=P, G=P, W=P, O=P, rms=None, B=4, H=256, D=128, eps=0.0, splits=0):
        return L.attn_rmsnorm_matmul(X, G, W, O, rms, B, H, D, eps, splits, None)
    assert rm(X=None) == 1
    assert rm(W=None) == 1
    assert rm(B=0) == 2
    assert rm(D=-8) == 2
    assert rm(H=100) == 3           # not a multiple of 8
    assert rm(D=12) == 3
    assert rm(eps=-1.0) == 8
    assert rm(eps=float("nan")) == 8
    assert rm(splits=3) == 8
    assert rm(splits=8, H=256) == 8  # only 4 K steps of 64
    assert rm(O=MIS) == 7
    assert rm(rms=ctypes.c_void_p(4098)) == 7
    def rmt(tile, splits=0):
        return L.attn_rmsnorm_matmul_tiled(P, P, P, P, None, 4, 256, 128, 0.0, tile, splits, None)
    assert rmt(24) == 8 and rmt(-16) == 8 and rmt(272) == 8
    assert L.attn_rmsnorm_matmul_splits(0, 64, 64) < 0
    S = L.attn_rmsnorm_matmul_splits(16, 4096, 4096)
    assert S in (1, 2, 4, 8)
    assert L.attn_rmsnorm_matmul_splits(1, 64, 8) == 1   # one K step


def test_rmsnorm_matmul_ws_validation_before_launch(L):
    """The workspace entry (two-pass form): form, workspace and its size are
    checked before anything reaches the device."""
    assert L.attn_rmsnorm_matmul_ws_bytes(0, 64) == 0
    assert L.attn_rmsnorm_matmul_ws_bytes(4, 256) == 2048 + 2 * 256   # X*G, then E and s
    need = L.attn_rmsnorm_matmul_ws_bytes(4, 256)

    def ws(form, work=P, nbytes=need, X=P, B=4, H=256, D=128):
        return L.attn_rmsnorm_matmul_ws(X, P, P, P, None, B, H, D, 0.0, form, work, nbytes, None)
    assert ws(3) == 8 and ws(-1) == 8            # unknown form
    assert ws(2, work=None) == 1                 # the two-pass form needs the workspace
    assert ws(2, nbytes=need - 16) == 4          # too small
    assert ws(2, work=MIS) == 7                  # misaligned
    assert ws(2, X=None) == 1
    assert ws(2, H=100) == 3                     # H not a multiple of 8
    assert ws(0, B=0) == 2 and ws(0, D=-8) == 2  # the automatic form checks shapes first
    assert ws(1, X=None) == 1                    # the fused form ignores the workspace
    assert ws(1, work=None, H=100) == 3


def test_prefill_splitkv_validation_before_launch(L):
    def sk(S, ws=P, wsb=1 << 30, Q=P):
        return L.attn_prefill_splitkv(Q, P, P, P, None, 1, 4, 2, 128, 128, 128, 1, 0.1, None, S,
                                      ws, wsb, None)
    assert sk(0) == 4 and sk(17) == 4
    assert sk(2, ws=None) == 1
    assert sk(2, Q=None) == 1
    assert sk(2, wsb=16) == 4
    assert sk(2, ws=MIS) == 7
    assert L.attn_prefill_splitkv_workspace_bytes(1, 4, 128, 128, 2) == 4 * 128 * 2 * 129 * 4
    assert L.attn_prefill_splitkv_workspace_bytes(1, 4, 128, 128, 1) == 0


def test_prefill_host_validation_before_copies(L):
    """Host-buffer prefill: every invalid argument is rejected before any copy
    or CUDA call (here no GPU exists, so reaching the device would give 5)."""
    opts = attn.PrefillOptions(1, 0.1, None, 0.0, -1, -1, 0)
    ws_need = L.attn_prefill_host_workspace_bytes(2, 8, 2, 100, 300, 128)
    # Q, K, V, O regions (256-byte aligned) and LSE
    rq = -(-2 * 8 * 100 * 128 * 2 // 256) * 256
    rkv = -(-2 * 2 * 300 * 128 * 2 // 256) * 256
    rl = -(-2 * 8 * 100 * 4 // 256) * 256
    assert ws_need == 2 * rq + 2 * rkv + rl
    assert L.attn_prefill_host_workspace_bytes(0, 8, 2, 100, 300, 128) == 0

    def call(Qh=P, Oh=P, B=2, Hq=8, Hkv=2, Lq=100, Lk=300, d=128, o=opts, ws=P, wsb=ws_need):
        return L.attn_prefill_host(Qh, P, P, Oh, None, B, Hq, Hkv, Lq, Lk, d,
                                   None if o is None else ctypes.byref(o), 0, ws, wsb, None)
    assert call(Qh=None) == 1
    assert call(Oh=None) == 1
    assert call(o=None) == 1
    assert call(ws=None) == 1
    assert call(Hq=6, Hkv=4) == 2
    assert call(Lq=0) == 2
    assert call(B=70000) == 2
    assert call(d=96) == 3
    assert call(o=attn.PrefillOptions(1, float("nan"), None, 0.0, -1, -1, 0)) == 8
    assert call(o=attn.PrefillOptions(1, 0.1, None, -1.0, -1, -1, 0)) == 8
    assert call(o=attn.PrefillOptions(1, 0.1, None, 0.0, -1, -1, 7)) == 3
    assert call(ws=MIS) == 7
    assert call(o=attn.PrefillOptions(1, 0.1, MIS.value, 0.0, -1, -1, 0)) == 7
    assert call(wsb=ws_need - 1) == 4


def test_prefill_host_chunking(L):
    """Chunks are runs of KV-head units inside one batch item, or whole batch
    items; automatic chunking aims at about 8 chunks."""
    assert L.attn_prefill_host_chunks(4, 32, 0) == 8       # 16 KV heads per chunk
    assert L.attn_prefill_host_chunks(4, 32, 8) == 16
    assert L.attn_prefill_host_chunks(4, 32, 5) == 4 * 7   # ragged last chunk per item
    assert L.attn_prefill_host_chunks(4, 32, 1) == 128
    assert L.attn_prefill_host_chunks(4, 32, 33) == 2      # rounded up to 2 whole items
    assert L.attn_prefill_host_chunks(5, 32, 64) == 3      # 2 + 2 + 1 items
    assert L.attn_prefill_host_chunks(64, 8, 0) == 8       # 8 whole items per chunk
    assert L.attn_prefill_host_chunks(1, 1, 0) == 1
    assert L.attn_prefill_host_chunks(0, 8, 0) == 0


def test_prefill_host_binding_rejects_device_tensors():
    q = torch.zeros(1, 2, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.prefill_host(q, q, q.float())
    with pytest.raises(TypeError):
        attn.prefill_host(None, q, q)
