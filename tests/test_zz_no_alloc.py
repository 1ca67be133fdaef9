"""GPU test of the allocation-free sequence entry point (gq4_run_sequence_static).

Two sequences in a row through the library's fixed scratch: a one-layer
7B-shaped decode chain (quad QKV, O, gated gate/up with its norm prologue,
down) and then the same chain again, each checked against the oracle on the
inputs the GPU produced, and bit for bit against gq4_run_sequence with a
caller workspace.  The library's plan query (gq4_sequence_launches) and,
where the profiler lists kernels, the kernel names show that the
persistent kernel (the one that uses the fixed scratch) ran; a chain of
more calls than one launch takes shows the array carried from one launch
to the next.
"""

import numpy as np
import pytest
import torch

import oracle
from int4_group_quantized_quant_gb300 import inputs as I
from tests.gpu_util import check_close, dev, gq4_module, host, requires_cuda, tol_fp32, tol_gated, wdev

pytestmark = [pytest.mark.gpu, requires_cuda]


def _nan(*shape):
    return torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")


def _layer(gq4, H, F, QKV, gs, seed):
    n0, n1, n2 = QKV[0], QKV[0] + QKV[1], sum(QKV)
    h = dev(I.activations(1, H, seed, 0))
    wqkv = I.quant_weights(H, n2, gs, seed, 1)
    wo = I.quant_weights(H, H, gs, seed, 2)
    wg = I.quant_weights(H, F, gs, seed, 3, scale_range=I.SCALE_RANGE_GATED)
    wu = I.quant_weights(H, F, gs, seed, 4, scale_range=I.SCALE_RANGE_GATED)
    wd = I.quant_weights(F, H, gs, seed, 5)
    W = dev(I.norm_gain(H, seed))
    q, k, v = _nan(1, QKV[0]), _nan(1, QKV[1]), _nan(1, QKV[2])
    o, res, f, hn = _nan(1, H), _nan(1, H), _nan(1, F), _nan(1, H)
    calls = [
        gq4.seq_quad(h, *wdev(wqkv), gs, n0, n1, n2, [q, k, v, None]),
        gq4.seq_matvec(q, *wdev(wo), gs, o),
        gq4.seq_gated(h, *wdev(wg), *wdev(wu), gs, f, W_norm=W, A_b=o, residual_out=res),
        gq4.seq_matvec(f, *wdev(wd), gs, hn),
    ]
    outs = dict(h=h, q=q, k=k, v=v, o=o, res=res, f=f, hn=hn, W=W)
    weights = dict(qkv=wqkv, o=wo, g=wg, u=wu, d=wd, splits=(n0, n1, n2))
    return calls, outs, weights


def _verify(outs, w, gs):
    n0, n1, n2 = w["splits"]
    ref, sabs = oracle.quad_matvec(host(outs["h"]), w["qkv"].Bq, w["qkv"].scales, w["qkv"].zeros,
                                   w["qkv"].K, w["qkv"].N, gs, n0, n1, n2)
    for i, name in enumerate(("q", "k", "v")):
        check_close(f"qkv out{i}", host(outs[name]), ref[i], tol_fp32(sabs[i]))
    C, S = oracle.matvec(host(outs["q"]), w["o"].Bq, w["o"].scales, w["o"].zeros, w["o"].K, w["o"].N, gs)
    check_close("o", host(outs["o"]), C, tol_fp32(S))
    r = oracle.gated_matvec(host(outs["h"]), w["g"].Bq, w["g"].scales, w["g"].zeros, w["u"].Bq,
                            w["u"].scales, w["u"].zeros, w["g"].K, w["g"].N, gs,
                            A_b=host(outs["o"]), W_norm=host(outs["W"]), eps=1e-6)
    check_close("gated", host(outs["f"]), r["out"], tol_gated(r["g"], r["u"], r["Sg"], r["Su"], r["out"]))
    assert np.array_equal(host(outs["res"]).view(np.uint32), r["residual_out"].view(np.uint32))
    C, S = oracle.matvec(host(outs["f"]), w["d"].Bq, w["d"].scales, w["d"].zeros, w["d"].K, w["d"].N, gs)
    check_close("down", host(outs["hn"]), C, tol_fp32(S))


def test_static_scratch_two_calls_in_a_row():
    gq4 = gq4_module()
    gq4.device_error(clear=True)
    calls, outs, w = _layer(gq4, 4096, 11008, (4096, 1024, 1024), 128, 1300)
    results = []
    for _ in range(2):
        for t in ("q", "k", "v", "o", "res", "f", "hn"):
            outs[t].fill_(float("nan"))
        gq4.run_sequence_static(calls)
        torch.cuda.synchronize()
        _verify(outs, w, 128)
        results.append(host(outs["hn"]).copy())
    assert np.array_equal(results[0].view(np.uint32), results[1].view(np.uint32))
    # the same bits as the caller-workspace entry point
    ws = gq4.sequence_workspace()
    gq4.run_sequence(calls, ws)
    torch.cuda.synchronize()
    assert np.array_equal(host(outs["hn"]).view(np.uint32), results[0].view(np.uint32))
    assert gq4.device_error() == 0


def _cuda_kernels(fn):
    """Names of the CUDA kernels run by fn(), from the profiler."""
    from torch.profiler import ProfilerActivity, profile
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    names = []
    for e in prof.events():
        if str(getattr(e, "device_type", "")).endswith("CUDA"):
            names.append(e.name)
    return names


def test_static_scratch_runs_the_persistent_kernel():
    gq4 = gq4_module()
    gq4.device_error(clear=True)
    calls, outs, w = _layer(gq4, 4096, 11008, (4096, 1024, 1024), 128, 1301)
    # the library's plan: one persistent launch (the kernel that uses the scratch)
    assert gq4.sequence_launches(calls) == 1
    names = _cuda_kernels(lambda: gq4.run_sequence_static(calls))
    if not names:
        pytest.skip("the profiler lists no CUDA kernels in this process")
    assert any("seq_kernel" in n for n in names), names
    assert not any("stream_matvec_kernel" in n for n in names), names
    _verify(outs, w, 128)
    assert gq4.device_error() == 0


def test_static_scratch_longer_than_one_launch():
    """133 chained small matvecs, h_{i+1} = W_i h_i, twice in a row: the
    second launch of each sequence reuses the array after the first one's
    exit reset, and the second sequence after the first's."""
    gq4 = gq4_module()
    gq4.device_error(clear=True)
    K, gs = 256, 64
    h = dev(I.activations(1, K, 1302))
    calls, chain = [], []
    for i in range(133):
        wi = I.quant_weights(K, K, gs, 1302, i, scale_range=(0.001, 0.004))
        nxt = _nan(1, K)
        calls.append(gq4.seq_matvec(h, *wdev(wi), gs, nxt))
        chain.append((h, wi, nxt))
        h = nxt
    # two persistent launches, the second reusing the array after the first's reset
    assert gq4.sequence_launches(calls) == 2
    finals = []
    for _ in range(2):
        for _, _, C in chain:
            C.fill_(float("nan"))
        gq4.run_sequence_static(calls)
        torch.cuda.synchronize()
        for i in (0, 1, 127, 128, 132):
            A, wi, C = chain[i]
            ref, S = oracle.matvec(host(A), wi.Bq, wi.scales, wi.zeros, K, K, gs)
            check_close(f"link {i}", host(C), ref, tol_fp32(S))
        finals.append(host(chain[-1][2]).copy())
    assert np.array_equal(finals[0].view(np.uint32), finals[1].view(np.uint32))
    assert gq4.device_error() == 0
