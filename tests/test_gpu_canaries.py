"""Out-of-bounds write checks with guard bands (a stand-in for a memory
sanitizer, which is not available on the GPUs these tests run on).

Every output of every kernel is carved out of a larger buffer: the bands
before and after it hold a sentinel bit pattern, the output itself is filled
with NaN. After a call on ragged shapes (query rows, keys and sequence
lengths that are not multiples of the kernels' tiles, empty sequences, rows
that see no key) the bands must be bit-for-bit unchanged and no NaN may be
left in the output: the kernel wrote every element it owns and nothing
outside. The small cases are also compared with the oracle.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention_ref, decode_ref, rmsnorm_matmul_ref
from tests.parity import assert_attention_close

pytestmark = pytest.mark.gpu

GUARD = 4096                 # elements per band; keeps the output 16-byte aligned
SENTINEL = {2: 0x5A5A, 4: 0x5A5A5A5A}


@pytest.fixture(scope="module")
def attn():
    import online_softmax_fusion_gb300 as m
    from online_softmax_fusion_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return m


class Guarded:
    """An output tensor with sentinel-filled bands on both sides."""

    def __init__(self, shape, dtype, scratch=False):
        self.n = int(math.prod(shape))
        self.buf = torch.empty(self.n + 2 * GUARD, dtype=dtype, device="cuda")
        self.size = self.buf.element_size()
        self._bits().fill_(SENTINEL[self.size])
        self.t = self.buf[GUARD:GUARD + self.n].view(shape)
        self.scratch = scratch      # a workspace: only the bands are checked
        if not scratch:
            self.t.fill_(float("nan"))

    def _bits(self):
        return self.buf.view(torch.int16 if self.size == 2 else torch.int32)

    def check(self, what):
        torch.cuda.synchronize()
        bits = self._bits()
        s = SENTINEL[self.size]
        lo = int((bits[:GUARD] != s).sum())
        hi = int((bits[GUARD + self.n:] != s).sum())
        assert lo == 0 and hi == 0, f"{what}: {lo} elements before and {hi} after it overwritten"
        if self.scratch:
            return
        nan = int(torch.isnan(self.t.float()).sum())
        assert nan == 0, f"{what}: {nan} elements never written (NaN left)"


def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


PREFILL_CASES = [
    # B, Hq, Hkv, Lq, Lk, d, causal
    (1, 2, 1, 1, 1, 128, False),       # one row, one key
    (1, 2, 2, 127, 65, 128, True),     # Lq < tile, Lk ragged
    (2, 2, 1, 129, 63, 64, True),      # Lq > Lk: leading rows see no key
    (1, 1, 1, 129, 1, 128, True),      # one key, most rows see none
    (1, 2, 2, 127, 200, 64, False),    # several key tiles, ragged tail
    (1, 4, 2, 257, 129, 128, True),    # GQA, two query heads per CTA
]


@pytest.mark.parametrize("impl", ["tcgen05", "tcgen05_1tile", "mma_sync"])
@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,d,causal", PREFILL_CASES)
def test_prefill_writes_exactly_its_output(attn, impl, B, Hq, Hkv, Lq, Lk, d, causal):
    q = _rand((B, Hq, Lq, d), Lq + 3 * Lk)
    k = _rand((B, Hkv, Lk, d), Lq + 3 * Lk + 1)
    v = _rand((B, Hkv, Lk, d), Lq + 3 * Lk + 2)
    O = Guarded((B, Hq, Lq, d), torch.bfloat16)
    L = Guarded((B, Hq, Lq), torch.float32)
    attn.prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, out=O.t, lse=L.t, impl=impl)
    O.check("O")
    L.check("LSE")
    assert attn.device_status() == 0
    Or, Lr = attention_ref(q, k, v, scale=d ** -0.5, causal=causal)
    assert_attention_close(O.t, L.t, Or, Lr)


@pytest.mark.parametrize("softcap,window", [(15.0, (-1, -1)), (0.0, (40, 7)), (20.0, (70, -1))])
def test_prefill_variants_write_exactly_their_output(attn, softcap, window):
    B, Hq, Hkv, Lq, Lk, d = 1, 4, 2, 131, 197, 128
    q = _rand((B, Hq, Lq, d), 61, 2.0)
    k = _rand((B, Hkv, Lk, d), 62, 2.0)
    v = _rand((B, Hkv, Lk, d), 63)
    O = Guarded((B, Hq, Lq, d), torch.bfloat16)
    L = Guarded((B, Hq, Lq), torch.float32)
    attn.prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, out=O.t, lse=L.t, softcap=softcap,
                 window=window)
    O.check("O")
    L.check("LSE")
    assert attn.device_status() == 0
    Or, Lr = attention_ref(q, k, v, scale=d ** -0.5, causal=True, softcap=softcap,
                           window_left=window[0], window_right=window[1])
    assert_attention_close(O.t, L.t, Or, Lr)


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,splits", [(1, 4, 2, 129, 65, 3), (2, 2, 2, 127, 300, 4),
                                                    (1, 2, 1, 200, 130, 2)])
def test_prefill_splitkv_writes_exactly_its_output(attn, B, Hq, Hkv, Lq, Lk, splits):
    d = 128
    q = _rand((B, Hq, Lq, d), 71 + Lq)
    k = _rand((B, Hkv, Lk, d), 72 + Lk)
    v = _rand((B, Hkv, Lk, d), 73 + Lk)
    nbytes = attn.lib().attn_prefill_splitkv_workspace_bytes(B, Hq, Lq, d, splits)
    ws = Guarded((nbytes // 4,), torch.float32)
    O = Guarded((B, Hq, Lq, d), torch.bfloat16)
    L = Guarded((B, Hq, Lq), torch.float32)
    attn.prefill_splitkv(q.cuda(), k.cuda(), v.cuda(), splits, causal=True, out=O.t, lse=L.t,
                         workspace=ws.t)
    O.check("O")
    L.check("LSE")
    # the partials: guarded; every one is written (empty splits with 0 / -inf)
    ws.check("split partials")
    assert attn.device_status() == 0
    Or, Lr = attention_ref(q, k, v, scale=d ** -0.5, causal=True)
    assert_attention_close(O.t, L.t, Or, Lr)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("S", [0, 3])
def test_decode_and_combine_write_exactly_their_outputs(attn, d, S):
    B, Hq, Hkv, Lmax = 4, 8, 2, 65
    lens = torch.tensor([0, 1, 63, 65], dtype=torch.int32)
    q = _rand((B, Hq, d), 81 + d)
    k = _rand((B, Hkv, Lmax, d), 82 + d)
    v = _rand((B, Hkv, Lmax, d), 83 + d)
    Sres = attn.resolve_splits(B, Hkv, Lmax, d, S)
    Op = Guarded((B, Hq, Sres, d), torch.float32)
    Lp = Guarded((B, Hq, Sres), torch.float32)
    attn.decode_splitk(q.cuda(), k.cuda(), v.cuda(), lens.cuda(), num_splits=Sres, o_part=Op.t,
                       lse_part=Lp.t)
    Op.check("O_part")
    Lp.check("LSE_part")
    O = Guarded((B, Hq, d), torch.bfloat16)
    L = Guarded((B, Hq), torch.float32)
    attn.combine(Op.t, Lp.t, out=O.t, lse=L.t)
    O.check("O")
    L.check("LSE")
    assert attn.device_status() == 0
    Or, Lr = decode_ref(q, k, v, lens, scale=d ** -0.5)
    assert_attention_close(O.t, L.t, Or, Lr)


def test_decode_noalloc_writes_exactly_its_output(attn):
    B, Hq, Hkv, Lmax, d = 3, 16, 2, 300, 128
    lens = torch.tensor([0, 129, 300], dtype=torch.int32)
    q = _rand((B, Hq, d), 91)
    k = _rand((B, Hkv, Lmax, d), 92)
    v = _rand((B, Hkv, Lmax, d), 93)
    O = Guarded((B, Hq, d), torch.bfloat16)
    L = Guarded((B, Hq), torch.float32)
    attn.decode_noalloc(q.cuda(), k.cuda(), v.cuda(), lens.cuda(), out=O.t, lse=L.t)
    O.check("O")
    L.check("LSE")
    assert attn.device_status() == 0
    Or, Lr = decode_ref(q, k, v, lens, scale=d ** -0.5)
    assert_attention_close(O.t, L.t, Or, Lr)


@pytest.mark.parametrize("impl,d", [("tcgen05", 128), ("mma_sync", 128), ("mma_sync", 64)])
@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk", [(1, 2, 1, 127, 127), (1, 2, 2, 129, 65),
                                            (2, 4, 2, 65, 200)])
def test_backward_writes_exactly_its_outputs(attn, impl, d, B, Hq, Hkv, Lq, Lk):
    q = _rand((B, Hq, Lq, d), 101 + Lq).cuda()
    k = _rand((B, Hkv, Lk, d), 102 + Lk).cuda()
    v = _rand((B, Hkv, Lk, d), 103 + Lk).cuda()
    do = _rand((B, Hq, Lq, d), 104).cuda()
    O, L = attn.prefill(q, k, v, causal=True)
    nbytes = attn.lib().attn_backward_workspace_bytes(B, Hq, Lq, d)
    ws = Guarded((nbytes // 4,), torch.float32)
    dq = Guarded(tuple(q.shape), torch.bfloat16)
    dk = Guarded(tuple(k.shape), torch.bfloat16)
    dv = Guarded(tuple(v.shape), torch.bfloat16)
    attn.backward(q, k, v, O, L, do, causal=True, workspace=ws.t, impl=impl, dq=dq.t, dk=dk.t,
                  dv=dv.t)
    for g, n in ((dq, "dQ"), (dk, "dK"), (dv, "dV"), (ws, "workspace")):
        g.check(n)
    assert attn.device_status() == 0


@pytest.mark.parametrize("form", [None, "two_pass"])
@pytest.mark.parametrize("B,H,D", [(5, 328, 200), (17, 136, 72), (3, 64, 64), (131, 200, 136)])
def test_rmsnorm_matmul_writes_exactly_its_outputs(attn, B, H, D, form):
    g = torch.Generator().manual_seed(B * 1000 + H)
    x = torch.randn(B, H, generator=g).to(torch.bfloat16)
    gw = (1 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    w = (torch.randn(H, D, generator=g) / H ** 0.5).to(torch.bfloat16)
    O = Guarded((B, D), torch.bfloat16)
    R = Guarded((B,), torch.float32)
    if form is None:
        attn.rmsnorm_matmul(x.cuda(), gw.cuda(), w.cuda(), out=O.t, rms=R.t)
    else:
        # the workspace is an output of the conversion pass: guarded too
        nbytes = attn.rmsnorm_matmul_ws_bytes(B, H)
        ws = Guarded((nbytes // 4,), torch.int32, scratch=True)
        attn.rmsnorm_matmul(x.cuda(), gw.cuda(), w.cuda(), out=O.t, rms=R.t, form=form,
                            workspace=ws.t)
        ws.check("workspace")
    O.check("O")
    R.check("RMS")
    assert attn.device_status() == 0
    ref = rmsnorm_matmul_ref(x, gw, w)
    s = float(np.sqrt(np.mean(ref * ref)))
    got = O.t.float().cpu().numpy()
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-2 * s)
