"""GPU parity of the fused attention forward (attention_bf16) against the CPU oracle:
O = softmax(scale * Q K^T) V per head, optionally causal.

Acceptance (oracle.check_attention): every element of O within
(2^-9 + 2e-4 + 1e-5 + 2e-5 * Ds) * (P|V|) + ulp_bf16(|O_ref|), the bound derived from the
BF16 rounding of the weights, FP32 accumulation and the score error.  Small problems are
compared in full; at full size every row of four heads of the batched shape and of the
causal 8192-token head, plus sampled query rows of every head.
"""
import numpy as np
import pytest

import oracle
import dense_gemm_sm_gb300 as dg
from dense_gemm_sm_gb300 import inputs

from .helpers import dev_bf16, host_bf16_bits, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = torch_mod()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    dg.load()
    return t


@pytest.fixture(params=["split", "nosplit"])
def split_mode(request, monkeypatch):
    # Key blocks split over CTAs (merged with the recurrence) when the query tiles do not
    # fill the GPU, or one CTA per query tile.
    if request.param == "nosplit":
        monkeypatch.setenv("DG_ATTN_SPLIT", "0")
    else:
        monkeypatch.delenv("DG_ATTN_SPLIT", raising=False)
    return request.param


def run(torch, w, O_fill=float("nan")):
    b, Lq = w["batch"], w["Lq"]
    n_out = (b - 1) * w["sO"] + (Lq - 1) * w["ldo"] + w["d"] if b > 0 and Lq > 0 else 1
    dO = torch.full((n_out,), O_fill, device="cuda", dtype=torch.bfloat16)
    dg.attention_bf16(b, Lq, w["Lkv"], w["d"], float(w["scale"]), w["causal"], dev_bf16(w["Q"]),
                      w["ldq"], w["sQ"], dev_bf16(w["K"]), w["ldk"], w["sK"], dev_bf16(w["V"]),
                      w["ldv"], w["sV"], dO, w["ldo"], w["sO"])
    torch.cuda.synchronize()
    assert dg.dg_device_status() == dg.DG_OK
    return host_bf16_bits(dO)


def gather(Ob, w, rows=None):
    """[batch, r, d] of O's bit patterns from the strided output buffer."""
    rows = np.arange(w["Lq"]) if rows is None else np.asarray(rows)
    idx = (np.arange(w["batch"])[:, None, None] * w["sO"] + rows[None, :, None] * w["ldo"] +
           np.arange(w["d"])[None, None, :])
    return Ob[idx]


def check(Ob, w, rows=None, what=""):
    O, PV, Ds = oracle.attention(w["batch"], w["Lq"], w["Lkv"], w["d"], float(w["scale"]),
                                 w["causal"], w["Q"], w["ldq"], w["sQ"], w["K"], w["ldk"], w["sK"],
                                 w["V"], w["ldv"], w["sV"], rows=rows)
    ok, worst = oracle.check_attention(gather(Ob, w, rows), O, PV, Ds)
    assert ok, f"{what}: error reaches {worst:.3g} x the bound"
    return worst


@pytest.mark.parametrize("batch,L,Lkv,causal", [
    (2, 256, 256, False),     # two query tiles, two key blocks
    (3, 300, 200, False),     # ragged query tile and key block
    (2, 384, 384, True),      # causal: 1..3 key blocks per query tile
    (1, 130, 130, True),      # causal with a 2-row last tile
    (2, 128, 1, False),       # one key: O = V[0]
    (1, 64, 1000, False),     # one partial query tile, eight key blocks
])
def test_attention_parity(torch, split_mode, batch, L, Lkv, causal):
    w = inputs.attention(batch, L, causal=causal, Lkv=Lkv)
    Ob = run(torch, w)
    check(Ob, w, what=f"attention b={batch} L={L} Lkv={Lkv} causal={causal}")
    if Lkv == 1:  # every weight is 1: O equals V's row exactly
        assert np.array_equal(gather(Ob, w)[:, :, :], np.broadcast_to(w["V"][:, :1, :], (batch, L, 128)))


def test_attention_large_score_spread(torch, split_mode):
    # Q scaled by 8: scores spread over ~+-90, so the reference maximum moves on many
    # blocks and the TMEM rescale of O runs; causal and non-causal.
    for causal in (False, True):
        w = inputs.attention(2, 1024, causal=causal, std_q=8.0)
        check(run(torch, w), w, what=f"attention spread causal={causal}")


def test_attention_padded_strides(torch):
    # Leading dimensions 136 and batch strides with gaps; the padding of O stays untouched.
    rng = np.random.default_rng(31)
    batch, L, d, ld = 3, 200, 128, 136
    stride = L * ld + 64
    mk = lambda: inputs.f32_to_bf16_bits(rng.normal(0, 1, batch * stride).astype(np.float32))
    w = dict(batch=batch, Lq=L, Lkv=L, d=d, causal=True, scale=np.float32(1 / np.sqrt(128.0)),
             Q=mk(), ldq=ld, sQ=stride, K=mk(), ldk=ld, sK=stride, V=mk(), ldv=ld, sV=stride,
             ldo=ld, sO=stride)
    Ob = run(torch, w)
    check(Ob, w, what="attention padded")
    written = np.zeros(Ob.shape, bool)
    idx = (np.arange(batch)[:, None, None] * stride + np.arange(L)[None, :, None] * ld +
           np.arange(d)[None, None, :])
    written[idx.reshape(-1)] = True
    assert np.all((Ob[~written] & 0x7FFF) > 0x7F80), "padding of O was written"


def head_view(w, h):
    """The single-head problem of head h of a strided batch (flat slices of Q, K and V)."""
    sl = lambda x, st: np.asarray(x).reshape(-1)[h * st: h * st + st] if st else x
    return dict(w, batch=1, Q=sl(w["Q"], w["sQ"]), K=sl(w["K"], w["sK"]), V=sl(w["V"], w["sV"]),
                sQ=0, sK=0, sV=0, sO=0)


def check_whole_head(Ob, w, h, what, rows_per_chunk=1024):
    """Every query row of head h against the oracle, in chunks of rows."""
    wh = head_view(w, h)
    Oh = Ob[h * w["sO"]: h * w["sO"] + (w["Lq"] - 1) * w["ldo"] + w["d"]] if w["sO"] else Ob
    for r0 in range(0, w["Lq"], rows_per_chunk):
        rows = np.arange(r0, min(w["Lq"], r0 + rows_per_chunk))
        check(Oh, wh, rows=rows, what=f"{what}, head {h}, rows {r0}..{rows[-1]}")


def test_attention_batched_full_size(torch):
    # The batched shape (64 heads x 2048 x 128, non-causal): every row of heads 0, 1, 32 and
    # 63 (the first and last head of each sequence's block of 32), and 48 sampled query rows
    # of every head, including the first and last of each 128-row tile edge.
    w = inputs.attention()
    Ob = run(torch, w)
    for h in (0, 1, 32, 63):
        check_whole_head(Ob, w, h, "attention 64x2048")
    rows = np.unique(np.concatenate([[0, 127, 128, 1023, 2047],
                                     np.random.default_rng(32).integers(0, 2048, 43)]))
    check(Ob, w, rows=rows, what="attention 64x2048 (sampled rows)")


def test_attention_causal_8k_whole(torch, split_mode):
    # One causal head of 8192 tokens (the pages' experiment), every query row, with and
    # without the split over keys.
    w = inputs.attention(1, 8192, causal=True)
    check_whole_head(run(torch, w), w, 0, "attention causal 8192")


def test_attention_deterministic(torch, split_mode):
    w = inputs.attention(4, 512, causal=True)
    outs = [run(torch, w) for _ in range(3)]
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_attention_errors(torch):
    t = torch.zeros(4 * 256 * 128, dtype=torch.bfloat16, device="cuda")
    f = dict(check=False)
    a = lambda *args: dg.attention_bf16(*args, **f)
    s = 0.088
    assert a(0, 128, 128, 128, s, 0, t, 128, 0, t, 128, 0, t, 128, 0, t, 128, 0) == dg.DG_OK
    assert a(1, 0, 128, 128, s, 0, t, 128, 0, t, 128, 0, t, 128, 0, t, 128, 0) == dg.DG_OK
    assert a(1, 128, 0, 128, s, 0, t, 128, 0, t, 128, 0, t, 128, 0, t, 128, 0) == dg.DG_ERR_INVALID_ARG
    assert a(-1, 128, 128, 128, s, 0, t, 128, 0, t, 128, 0, t, 128, 0, t, 128, 0) == dg.DG_ERR_INVALID_ARG
    assert a(1, 128, 128, 64, s, 0, t, 64, 0, t, 64, 0, t, 64, 0, t, 64, 0) == dg.DG_ERR_UNSUPPORTED
    assert a(1, 128, 128, 128, 0.0, 0, t, 128, 0, t, 128, 0, t, 128, 0, t, 128, 0) == dg.DG_ERR_INVALID_ARG
    assert a(1, 128, 128, 128, float("inf"), 0, t, 128, 0, t, 128, 0, t, 128, 0, t, 128, 0) == dg.DG_ERR_INVALID_ARG
    assert a(1, 128, 64, 128, s, 1, t, 128, 0, t, 128, 0, t, 128, 0, t, 128, 0) == dg.DG_ERR_INVALID_ARG
    assert a(1, 128, 128, 128, s, 0, t, 120, 0, t, 128, 0, t, 128, 0, t, 128, 0) == dg.DG_ERR_INVALID_ARG
    assert a(2, 128, 128, 128, s, 0, t, 128, 128 * 128, t, 128, 128 * 128, t, 128, 128 * 128,
             t, 128, 100 * 128) == dg.DG_ERR_INVALID_ARG          # overlapping O batches
    assert a(1, 128, 128, 128, s, 0, t, 132, 0, t, 128, 0, t, 128, 0, t, 128, 0) == dg.DG_ERR_MISALIGNED
    assert a(1, 128, 128, 128, s, 0, t.data_ptr() + 2, 128, 0, t, 128, 0, t, 128, 0, t, 128,
             0) == dg.DG_ERR_MISALIGNED


@pytest.mark.parametrize("batch,L,Lkv", [(152, 256, 256), (160, 300, 200), (100, 512, 1000)])
def test_attention_two_tile_kernel(torch, batch, L, Lkv):
    # The opt-in two-tile kernel (DG_ATTN_PAIR=1) with enough query tiles that each CTA takes
    # a pair: ragged query and key lengths, a last pair with only one tile; compared in
    # full, and bit for bit with the default one-tile kernel (the same operations per row in
    # the same order).
    import os
    w = inputs.attention(batch, L, Lkv=Lkv)
    os.environ["DG_ATTN_PAIR"] = "1"
    try:
        Ob = run(torch, w)
    finally:
        del os.environ["DG_ATTN_PAIR"]
    check(Ob, w, what=f"attention two-tile b={batch} L={L} Lkv={Lkv}")
    Ob1 = run(torch, w)
    assert np.array_equal(Ob, Ob1)
