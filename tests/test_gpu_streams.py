"""The backward's side stream: dweight runs beside dhidden on an internal stream forked from
the caller's stream and joined back before the call returns.  Results must not depend on
which stream the caller uses, work the caller enqueues after the call must see the
finished gradients, and concurrent calls from two host threads on their own streams (each
thread has its own side stream) must each be right."""
import dataclasses
import threading

import pytest
import torch

from linear_cross_entropy_forward_gb300 import (flce_backward, flce_forward,
                                                flce_forward_backward)
from linear_cross_entropy_forward_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

W = dataclasses.replace(wl.TINY, name="st", N=1100, H=200, V=1000, reduction="none",
                        grad_mode="normal", zloss_coef=1e-3)


def _cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_cross_entropy_forward_gb300.build import build
    build()


def _inputs(seed=0):
    w = dataclasses.replace(W, seed=seed)
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(w)
    dev = torch.device("cuda")
    return (hidden.to(dev), weight.to(dev), labels.to(dev), g_loss.to(dev), g_ent.to(dev))


def _two_call(hd, Wd, yd, gl, ge, chunk_v):
    _, _, lse, ez = flce_forward(hd, Wd, yd, "none", zloss_coef=1e-3, validate=True)
    return flce_backward(hd, Wd, yd, lse, ez, gl, ge, "none", zloss_coef=1e-3, validate=True,
                         chunk_v=chunk_v)


def _bits(t):
    return t.view(torch.int16)


@pytest.mark.parametrize("chunk_v", [0, 256])
def test_user_stream_gives_the_default_streams_bits(chunk_v):
    _cuda_or_skip()
    hd, Wd, yd, gl, ge = _inputs()
    ref = _two_call(hd, Wd, yd, gl, ge, chunk_v)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dh, dw = _two_call(hd, Wd, yd, gl, ge, chunk_v)
        # enqueued after the call on the same stream: must see the finished gradients
        dw_copy = dw.clone()
        dh_copy = dh.clone()
    s.synchronize()
    assert torch.equal(_bits(dh), _bits(ref[0])) and torch.equal(_bits(dw), _bits(ref[1]))
    assert torch.equal(_bits(dh_copy), _bits(ref[0]))
    assert torch.equal(_bits(dw_copy), _bits(ref[1]))


def test_gradient_in_forward_on_a_user_stream():
    _cuda_or_skip()
    hd, Wd, yd, gl, ge = _inputs()
    ref = flce_forward_backward(hd, Wd, yd, gl, ge, "none", zloss_coef=1e-3, chunk_n=512)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = flce_forward_backward(hd, Wd, yd, gl, ge, "none", zloss_coef=1e-3, chunk_n=512)
        dw_copy = out[5].clone()
    s.synchronize()
    assert torch.equal(_bits(out[4]), _bits(ref[4])) and torch.equal(_bits(out[5]), _bits(ref[5]))
    assert torch.equal(_bits(dw_copy), _bits(ref[5]))


def test_two_host_threads_on_their_own_streams():
    _cuda_or_skip()
    inputs = [_inputs(seed) for seed in (0, 1)]
    refs = []
    for args in inputs:
        refs.append(_two_call(*args, chunk_v=256))
    torch.cuda.synchronize()
    results = [None, None]
    errors = []

    def work(i):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                outs = []
                for _ in range(3):
                    outs.append(_two_call(*inputs[i], chunk_v=256))
            s.synchronize()
            results[i] = outs
        except Exception as e:  # reported in the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    for i in range(2):
        for dh, dw in results[i]:
            assert torch.equal(_bits(dh), _bits(refs[i][0]))
            assert torch.equal(_bits(dw), _bits(refs[i][1]))


def test_thread_exit_with_the_backward_still_running():
    """A host thread that enqueues a backward and exits at once: its side stream and
    events are destroyed at thread exit while dweight may still be running on them,
    which must neither lose nor reorder work."""
    _cuda_or_skip()
    args = _inputs(0)
    ref = _two_call(*args, chunk_v=256)
    torch.cuda.synchronize()
    for _ in range(4):
        box = {}

        def work():
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            hd, Wd, yd, gl, ge = args
            with torch.cuda.stream(s):
                # without validate nothing waits for the stream before the thread ends
                _, _, lse, ez = flce_forward(hd, Wd, yd, "none", zloss_coef=1e-3)
                box["out"] = flce_backward(hd, Wd, yd, lse, ez, gl, ge, "none",
                                           zloss_coef=1e-3, chunk_v=256)
            box["stream"] = s

        t = threading.Thread(target=work)
        t.start()
        t.join(timeout=120)
        assert "out" in box
        box["stream"].synchronize()
        dh, dw = box["out"]
        assert torch.equal(_bits(dh), _bits(ref[0]))
        assert torch.equal(_bits(dw), _bits(ref[1]))


def _mixed_case(i):
    import random
    r = random.Random(95000 + i)
    layout = r.choice(["hv", "vh"])
    V = r.randint(1, 6000) if layout == "vh" else 8 * r.randint(1, 750)
    red = r.choice(["mean", "sum", "none"])
    w = dataclasses.replace(wl.TINY, name=f"c{i}", seed=950 + i,
                            N=r.choice([1, 37, 300, 1100, 2500]), H=8 * r.randint(1, 96), V=V,
                            reduction=red, zloss_coef=r.choice([0.0, 1e-3]),
                            softcap=r.choice([0.0, 5.0]),
                            grad_mode="normal" if red == "none" else "ones")
    h, W, y, gl, ge = wl.make_inputs(w)
    if layout == "vh":
        W = W.t().contiguous()
    dev = torch.device("cuda")
    return (w, tuple(x.to(dev) for x in (h, W, y, gl, ge)),
            dict(zloss_coef=w.zloss_coef, softcap=w.softcap, weight_layout=layout),
            r.random() < 0.4, r.choice([0, 256, 1024]))


def _run_mixed(w, t, kw, gif, chunk_v):
    hd, Wd, yd, gl, ge = t
    if gif:
        return flce_forward_backward(hd, Wd, yd, gl, ge, w.reduction, **kw)
    loss, ent, lse, ez = flce_forward(hd, Wd, yd, w.reduction, **kw)
    dh, dw = flce_backward(hd, Wd, yd, lse, ez, gl, ge, w.reduction, chunk_v=chunk_v, **kw)
    return loss, ent, lse, ez, dh, dw


def test_four_host_threads_with_mixed_problems():
    """Four host threads, each on its own stream, run a shuffled mix of problems (both
    layouts, both modes, several chunkings) twice over; every result must be bitwise
    the one the same call gives alone (the per-device caches, side streams and tile
    counters shared by concurrent calls must not leak between them)."""
    _cuda_or_skip()
    cases = [_mixed_case(i) for i in range(8)]
    refs = [[x.clone() for x in _run_mixed(*c)] for c in cases]
    torch.cuda.synchronize()
    fails = []

    def work(tid):
        import random
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            order = list(range(len(cases)))
            random.Random(tid).shuffle(order)
            with torch.cuda.stream(s):
                for _ in range(2):
                    for k in order:
                        out = _run_mixed(*cases[k])
                        s.synchronize()
                        for a, b in zip(out, refs[k]):
                            if not torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16
                                               else a,
                                               b.view(torch.int16) if b.dtype == torch.bfloat16
                                               else b):
                                fails.append((tid, k))
                                break
        except Exception as e:  # reported in the main thread
            fails.append((tid, repr(e)))

    threads = [threading.Thread(target=work, args=(t,)) for t in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not fails, fails
