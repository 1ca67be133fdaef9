"""GPU parity of one-lane call sequences (gq4_run_sequence).

A sequence runs its calls in order in one persistent launch; call i+1 may
read what calls 0..i wrote.  Every intermediate here has a buffer of its own,
filled with NaN before the run, so after the run each call is checked
against the oracle on the very inputs the GPU produced for it: a call that
read a stale or unwritten input fails.  Cases: two 7B-shaped decode layers
(quad QKV, O, gated gate/up with its norm prologue, down), every op with
ragged column counts and group sizes 32..256, a sequence longer than one
launch holds, scale rows that are not 16-byte aligned (run as individual
launches), workspace reuse and determinism.
"""

import numpy as np
import pytest
import torch

import oracle
from int4_group_quantized_quant_gb300 import inputs as I
from tests.gpu_util import check_close, dev, gq4_module, host, requires_cuda, tol_fp32, tol_gated, wdev

pytestmark = [pytest.mark.gpu, requires_cuda]


@pytest.fixture(scope="module")
def gq4():
    g = gq4_module()
    g.device_error(clear=True)
    return g


def _nan(*shape):
    return torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")


def _check_matvec(name, C, A, w, gs):
    ref, S = oracle.matvec(host(A), w.Bq, w.scales, w.zeros, w.K, w.N, gs)
    check_close(name, host(C), ref, tol_fp32(S))


def _check_gated(name, out, A, wg, wu, gs, A_b=None, W=None, res=None):
    kw = {}
    if W is not None:
        kw = dict(A_b=host(A_b), W_norm=host(W), eps=1e-6)
    r = oracle.gated_matvec(host(A), wg.Bq, wg.scales, wg.zeros, wu.Bq, wu.scales, wu.zeros,
                            wg.K, wg.N, gs, **kw)
    check_close(name, host(out), r["out"], tol_gated(r["g"], r["u"], r["Sg"], r["Su"], r["out"]))
    if res is not None:
        assert np.array_equal(host(res).view(np.uint32), r["residual_out"].view(np.uint32)), name


def _layers(gq4, n_layers, H, F, QKV, gs, seed):
    """Calls and buffers of n_layers decode layers, every intermediate distinct."""
    nq = sum(QKV)
    n0, n1, n2 = QKV[0], QKV[0] + QKV[1], nq
    h = dev(I.activations(1, H, seed, 0))
    calls, checks = [], []
    for li in range(n_layers):
        wqkv = I.quant_weights(H, nq, gs, seed, li, 1)
        wo = I.quant_weights(H, H, gs, seed, li, 2)
        wg = I.quant_weights(H, F, gs, seed, li, 3, scale_range=I.SCALE_RANGE_GATED)
        wu = I.quant_weights(H, F, gs, seed, li, 4, scale_range=I.SCALE_RANGE_GATED)
        wd = I.quant_weights(F, H, gs, seed, li, 5)
        W = dev(I.norm_gain(H, seed, li))
        q, k, v = _nan(1, QKV[0]), _nan(1, QKV[1]), _nan(1, QKV[2])
        o, res, f, hn = _nan(1, H), _nan(1, H), _nan(1, F), _nan(1, H)
        calls += [
            gq4.seq_quad(h, *wdev(wqkv), gs, n0, n1, n2, [q, k, v, None]),
            gq4.seq_matvec(q, *wdev(wo), gs, o),
            gq4.seq_gated(h, *wdev(wg), *wdev(wu), gs, f, W_norm=W, A_b=o, residual_out=res),
            gq4.seq_matvec(f, *wdev(wd), gs, hn),
        ]
        checks.append((h, wqkv, q, k, v, wo, o, wg, wu, W, res, f, wd, hn, (n0, n1, n2)))
        h = hn
    return calls, checks


def _verify_layers(checks, gs):
    for li, (h, wqkv, q, k, v, wo, o, wg, wu, W, res, f, wd, hn, splits) in enumerate(checks):
        n0, n1, n2 = splits
        outs_ref, sabs = oracle.quad_matvec(host(h), wqkv.Bq, wqkv.scales, wqkv.zeros, wqkv.K,
                                            wqkv.N, gs, n0, n1, n2)
        for i, t in enumerate((q, k, v)):
            check_close(f"layer {li} qkv out{i}", host(t), outs_ref[i], tol_fp32(sabs[i]))
        _check_matvec(f"layer {li} o", o, q, wo, gs)
        _check_gated(f"layer {li} gated", f, h, wg, wu, gs, A_b=o, W=W, res=res)
        _check_matvec(f"layer {li} down", hn, f, wd, gs)


def test_seq_two_decode_layers(gq4):
    """Two 7B-shaped layers: hidden 4096, ffn 11008, qkv 4096+1024+1024, group 128."""
    calls, checks = _layers(gq4, 2, 4096, 11008, (4096, 1024, 1024), 128, 1200)
    ws = gq4.sequence_workspace()
    gq4.run_sequence(calls, ws)
    torch.cuda.synchronize()
    _verify_layers(checks, 128)
    assert gq4.device_error() == 0
    assert int(ws[:4].view(torch.int32).item()) == 0  # arrival counter back at zero


def test_seq_small_layers_group_32(gq4):
    """Three small layers at group size 32 (one-chunk groups) and ragged widths."""
    calls, checks = _layers(gq4, 3, 512, 1344, (512, 96, 96), 32, 1201)
    ws = gq4.sequence_workspace()
    gq4.run_sequence(calls, ws)
    torch.cuda.synchronize()
    _verify_layers(checks, 32)
    assert gq4.device_error() == 0


def test_seq_every_op_ragged(gq4):
    """Each op once, with column counts that leave partial warp slots and ring
    entries, group sizes 32..256 (43 groups per column: scale rows start
    16-byte aligned only every 4 columns); the gated call reads the norm
    call's residual_out."""
    K1, N1, gs1 = 2560, 1001, 64
    w1 = I.quant_weights(K1, N1, gs1, 1202, 1)
    A = dev(I.activations(1, K1, 1202))
    C1 = _nan(1, N1)
    K2, N2, gs2 = 11008, 77, 256
    w2 = I.quant_weights(1024, 3, 32, 1202, 2)
    A2 = dev(I.activations(1, 1024, 1202, 3))
    Ab2 = dev(I.activations(1, 1024, 1202, 4))
    W2 = dev(I.norm_gain(1024, 1202))
    C2, res2, nout2 = _nan(1, 3), _nan(1, 1024), _nan(1, 1024)
    w3 = I.quant_weights(K2, N2, gs2, 1202, 5)
    A3 = dev(I.activations(1, K2, 1202, 5))
    outs3 = [_nan(1, 10), _nan(1, 0), _nan(1, 60), _nan(1, 7)]
    wg = I.quant_weights(1024, 131, 128, 1202, 6, scale_range=I.SCALE_RANGE_GATED)
    wu = I.quant_weights(1024, 131, 128, 1202, 7, scale_range=I.SCALE_RANGE_GATED)
    out4 = _nan(1, 131)
    calls = [
        gq4.seq_matvec(A, *wdev(w1), gs1, C1),
        gq4.seq_norm(A2, *wdev(w2), 32, W2, C2, A_b=Ab2, residual_out=res2, norm_out=nout2),
        gq4.seq_quad(A3, *wdev(w3), gs2, 10, 10, 70, [outs3[0], None, outs3[2], outs3[3]]),
        gq4.seq_gated(res2, *wdev(wg), *wdev(wu), 128, out4),
    ]
    ws = gq4.sequence_workspace()
    gq4.run_sequence(calls, ws)
    torch.cuda.synchronize()
    _check_matvec("matvec", C1, A, w1, gs1)
    ref, S, res_ref, nout_ref = oracle.norm_matvec(host(A2), host(Ab2), host(W2), 1e-6, w2.Bq,
                                                   w2.scales, w2.zeros, 1024, 3, 32)
    check_close("norm", host(C2), ref, tol_fp32(S))
    assert np.array_equal(host(res2).view(np.uint32), res_ref.view(np.uint32))
    check_close("norm_out", host(nout2), nout_ref, 1e-5 * np.abs(nout_ref) + 1e-7)
    outs_ref, sabs = oracle.quad_matvec(host(A3), w3.Bq, w3.scales, w3.zeros, K2, N2, gs2, 10, 10, 70)
    for i in (0, 2, 3):
        check_close(f"quad out{i}", host(outs3[i]), outs_ref[i], tol_fp32(sabs[i]))
    _check_gated("gated over the norm call's residual_out", out4, res2, wg, wu, 128)
    assert gq4.device_error() == 0


def test_seq_longer_than_one_launch(gq4):
    """133 chained small matvecs (more than one launch takes): h_{i+1} = W_i h_i."""
    K, gs = 256, 64
    h = dev(I.activations(1, K, 1203))
    calls, chain = [], []
    for i in range(133):
        w = I.quant_weights(K, K, gs, 1203, i, scale_range=(0.001, 0.004))
        nxt = _nan(1, K)
        calls.append(gq4.seq_matvec(h, *wdev(w), gs, nxt))
        chain.append((h, w, nxt))
        h = nxt
    ws = gq4.sequence_workspace()
    gq4.run_sequence(calls, ws)
    torch.cuda.synchronize()
    for i in (0, 1, 63, 64, 127, 128, 132):
        A, w, C = chain[i]
        _check_matvec(f"link {i}", C, A, w, gs)
    assert gq4.device_error() == 0


def test_seq_unaligned_rows_run_individually(gq4):
    """Scale rows 4 bytes past a 16-byte boundary: the calls run one by one,
    same semantics (the second reads the first's output)."""
    K, N, gs = 1024, 1024, 128
    w1 = I.quant_weights(K, N, gs, 1204, 1)
    w2 = I.quant_weights(N, 300, gs, 1204, 2)
    flat = torch.zeros(w1.scales.size + 8, dtype=torch.float32, device="cuda")
    s1 = flat[1:1 + w1.scales.size].view(*w1.scales.shape)
    s1.copy_(torch.from_numpy(w1.scales).cuda())
    A = dev(I.activations(1, K, 1204))
    C1, C2 = _nan(1, N), _nan(1, 300)
    Bq1, _, z1 = wdev(w1)
    calls = [gq4.seq_matvec(A, Bq1, s1, z1, gs, C1), gq4.seq_matvec(C1, *wdev(w2), gs, C2)]
    ws = gq4.sequence_workspace()
    gq4.run_sequence(calls, ws)
    torch.cuda.synchronize()
    _check_matvec("first", C1, A, w1, gs)
    _check_matvec("second", C2, C1, w2, gs)


def test_seq_reuse_and_determinism(gq4):
    """The same workspace serves consecutive sequences; results repeat bit for bit."""
    calls, checks = _layers(gq4, 1, 1024, 2816, (1024, 256, 256), 128, 1205)
    ws = gq4.sequence_workspace()
    outs = []
    for _ in range(3):
        gq4.run_sequence(calls, ws)
        torch.cuda.synchronize()
        outs.append(host(checks[0][13]).copy())
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert np.array_equal(outs[0].view(np.uint32), outs[2].view(np.uint32))
    _verify_layers(checks, 128)
    assert gq4.device_error() == 0
