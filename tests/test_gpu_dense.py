"""GPU parity of the output layer (lm_head) and the dense FFN layers against the C++ oracle.

Both are one streaming NVFP4 GEMV on the tensor cores with exact products, so
they differ from the oracle only in the order of fp32 additions:

* logits: every element within Higham's bound gamma_K * sum_k |w_k x_k| (plus
  2 ulp for the tensor-scale product) of the oracle's, and the arg-max token
  the same wherever the oracle's top two logits are further apart than that;
* dense FFN: bf16 outputs within the decode tolerances (relative L2 1e-3,
  max-abs 2e-2 x RMS of the oracle's bf16-rounded output), with and without
  the residual.

Sizes: tiny shapes (several row tiles, several K slices, ragged token counts,
more than one 32-token pass) and the Flint readings (vocab 151,936 x 2048;
d_ff 18,432).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import cpp
from tests import harness

pytestmark = pytest.mark.gpu
U = 2.0 ** -24


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_expert_ffn_gemv_b300 as lib
    return lib


def _quantized(lib, w):
    c, s, ts = lib.quantize(w.cuda())
    return dict(codes=c, scales=s, tensor_scale=ts)


def _head(lib, vocab, d, max_tokens, seed):
    w = synth.head_weight(vocab, d, seed, device="cuda")
    m = _quantized(lib, w)
    ctx = lib.moe_head_init(vocab, d, m, max_tokens)
    oc, os_, ots = cpp.quantize(w.cpu().numpy())
    return ctx, (oc, os_, ots)


def _check_logits(got, x, oracle_w):
    oc, os_, ots = oracle_w
    ref = cpp.gemv(oc, os_, ots, x).astype(np.float64)
    wq = np.abs(cpp.dequantize(oc, os_, ots).astype(np.float64))
    bound = (x.shape[1] * U / (1 - x.shape[1] * U)) * (np.abs(x.astype(np.float64)) @ wq.T) + 2 * U * np.abs(ref)
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= bound + 1e-30), f"logit error {np.max(err / (bound + 1e-30)):.2f} x the bound"
    top2 = -np.sort(-ref, axis=1)[:, :2]
    clear = (top2[:, 0] - top2[:, 1]) > 2 * np.max(bound, axis=1)
    assert np.array_equal(np.argmax(got, axis=1)[clear], np.argmax(ref, axis=1)[clear])


@pytest.mark.parametrize("T", [1, 5, 33])
def test_head_small(lib, T):
    vocab, d = 400, 256
    ctx, ow = _head(lib, vocab, d, 64, seed=7)
    try:
        xb, x = synth.tokens(synth.MoEShape(d, 1, 1, 128), T, seed=500 + T)
        out = torch.empty((T, vocab), dtype=torch.float32, device="cuda")
        lib.moe_head_forward(ctx, xb.cuda(), T, out)
        assert lib.moe_dense_get_device_status(ctx) == 0
        _check_logits(out.cpu().numpy(), x.numpy(), ow)
    finally:
        lib.moe_dense_destroy(ctx)


@pytest.mark.parametrize("d", [1024, 2048])
def test_head_one_token_fma_path(lib, d):
    """One token at d_model 1024 or 2048 takes the FMA consumer (x in registers); 33 tokens end
    with a one-token pass at offset 32, through the same consumer."""
    vocab = 1008
    ctx, ow = _head(lib, vocab, d, 64, seed=11)
    try:
        for T in (1, 33):
            xb, x = synth.tokens(synth.MoEShape(d, 1, 1, 128), T, seed=600 + T)
            out = torch.empty((T, vocab), dtype=torch.float32, device="cuda")
            lib.moe_head_forward(ctx, xb.cuda(), T, out)
            assert lib.moe_dense_get_device_status(ctx) == 0
            _check_logits(out.cpu().numpy(), x.numpy(), ow)
    finally:
        lib.moe_dense_destroy(ctx)


def test_head_flint(lib):
    vocab, d = synth.FLINT_VOCAB, synth.FLINT.d_model
    ctx, ow = _head(lib, vocab, d, 8, seed=synth.head_seed())
    try:
        for T in (1, 3):
            xb, x = synth.tokens(synth.FLINT, T, seed=synth.token_seed(600 + T))
            out = torch.empty((T, vocab), dtype=torch.float32, device="cuda")
            lib.moe_head_forward(ctx, xb.cuda(), T, out)
            assert lib.moe_dense_get_device_status(ctx) == 0
            _check_logits(out.cpu().numpy(), x.numpy(), ow)
    finally:
        lib.moe_dense_destroy(ctx)


def _ffn(lib, d, f, max_tokens, seed):
    wg, wu, wd = synth.dense_ffn_weights(d, f, seed, device="cuda")
    mg, mu, md = (_quantized(lib, w) for w in (wg, wu, wd))
    ctx = lib.moe_ffn_init(d, f, mg, mu, md, max_tokens)
    oracle = tuple(cpp.quantize(w.cpu().numpy()) for w in (wg, wu, wd))
    return ctx, oracle


def _check_ffn(lib, ctx, oracle, shape, T, seed, residual):
    xb, x = synth.tokens(shape, T, seed=seed)
    y = torch.empty((T, shape.d_model), dtype=torch.bfloat16, device="cuda")
    lib.moe_ffn_forward(ctx, xb.cuda(), T, y, residual)
    assert lib.moe_dense_get_device_status(ctx) == 0
    ref = cpp.dense_ffn(*oracle, x.numpy())
    want = cpp.residual(x.numpy(), ref) if residual else cpp.bf16_rne(ref)
    return harness.assert_close(y, want, f"dense FFN T={T} residual={residual}")


@pytest.mark.parametrize("T", [1, 7, 40])
def test_dense_ffn_small(lib, T):
    d, f = 256, 4608          # two K slices of 2304 in the down projection (MMA consumers at every T)
    shape = synth.MoEShape(d, 1, 1, 128)
    ctx, oracle = _ffn(lib, d, f, 64, seed=9)
    try:
        _check_ffn(lib, ctx, oracle, shape, T, seed=700 + T, residual=0)
        _check_ffn(lib, ctx, oracle, shape, T, seed=800 + T, residual=1)
    finally:
        lib.moe_dense_destroy(ctx)


@pytest.mark.parametrize("T", [1, 33])
def test_dense_ffn_one_token_fma_paths(lib, T):
    """d_model 1024 and 2048-wide K slices: one token takes the FMA consumers of both passes (h read
    as fp32 by the down pass, no hi / lo split); 33 tokens run a 32-token MMA pass, then a one-token
    pass at offset 32 through the FMA consumers."""
    d, f = 1024, 4096         # two K slices of 2048 in the down projection
    shape = synth.MoEShape(d, 1, 1, 128)
    ctx, oracle = _ffn(lib, d, f, 64, seed=13)
    try:
        _check_ffn(lib, ctx, oracle, shape, T, seed=900 + T, residual=0)
        _check_ffn(lib, ctx, oracle, shape, T, seed=950 + T, residual=1)
    finally:
        lib.moe_dense_destroy(ctx)


def test_dense_ffn_flint(lib):
    d, f = synth.FLINT.d_model, synth.FLINT_DENSE_FF
    ctx, oracle = _ffn(lib, d, f, 8, seed=synth.dense_seed(0))
    try:
        for T, res in ((1, 0), (1, 1), (5, 1)):
            _check_ffn(lib, ctx, oracle, synth.FLINT, T, seed=synth.token_seed(900 + T), residual=res)
    finally:
        lib.moe_dense_destroy(ctx)


@pytest.mark.parametrize("T", [1, 8])
def test_dense_chain_back_to_back_matches_synchronised(lib, T):
    """Dense FFN layers feeding each other, then the output layer, queued back to back: each
    forward's first kernels may start (programmatic dependent launch) while the previous forward
    still runs.  The results equal, bit for bit, those of the same chain with a synchronisation
    after every forward."""
    d, f, vocab = 1024, 4096, 400
    shape = synth.MoEShape(d, 1, 1, 128)
    ffns = [_ffn(lib, d, f, 64, seed=20 + i)[0] for i in range(3)]
    head, _ = _head(lib, vocab, d, 64, seed=23)
    try:
        xb, _ = synth.tokens(shape, T, seed=990 + T)

        def run(sync):
            cur = xb.cuda()
            for c in ffns:
                y = torch.empty_like(cur)
                lib.moe_ffn_forward(c, cur, T, y, 1)
                if sync:
                    torch.cuda.synchronize()
                cur = y
            logits = torch.empty((T, vocab), dtype=torch.float32, device="cuda")
            lib.moe_head_forward(head, cur, T, logits)
            torch.cuda.synchronize()
            return cur.view(torch.int16).cpu(), logits.view(torch.int32).cpu()

        a, b = run(False), run(True)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
        for c in ffns + [head]:
            assert lib.moe_dense_get_device_status(c) == 0
    finally:
        for c in ffns + [head]:
            lib.moe_dense_destroy(c)


def test_dense_kernel_counts(lib):
    """The launches a forward makes, as the library reports them for accounting: 2 per 32-token
    pass of the output layer; 5 per dense FFN pass, 4 for a one-token pass with 2048-wide K slices."""
    head, _ = _head(lib, 400, 256, 64, seed=7)
    ffn_2048, _ = _ffn(lib, 1024, 4096, 64, seed=13)
    ffn_2304, _ = _ffn(lib, 256, 4608, 64, seed=9)
    try:
        assert [lib.moe_dense_kernels_per_forward(head, T) for T in (0, 1, 32, 33)] == [0, 2, 2, 4]
        assert [lib.moe_dense_kernels_per_forward(ffn_2048, T) for T in (1, 2, 33)] == [4, 5, 9]
        assert [lib.moe_dense_kernels_per_forward(ffn_2304, T) for T in (1, 33)] == [5, 10]
    finally:
        for c in (head, ffn_2048, ffn_2304):
            lib.moe_dense_destroy(c)


def test_dense_rejects_bad_arguments(lib):
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    m = dict(codes=z, scales=z, tensor_scale=torch.zeros(1, device="cuda"))
    for bad in ((400, 300), (401, 256)):     # d_model not a power of two; vocab not a multiple of 16
        with pytest.raises(lib.MoEError):
            lib.moe_head_init(bad[0], bad[1], m, 4)
    with pytest.raises(lib.MoEError):
        lib.moe_ffn_init(256, 200, m, m, m, 4)   # d_ff not a multiple of 256
