"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
symbol include/flce.h declares, sizes workspaces and rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

import linear_cross_entropy_forward_gb300 as flce
from linear_cross_entropy_forward_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flce.h")


@pytest.fixture(scope="module")
def lib():
    from linear_cross_entropy_forward_gb300.build import build
    build()
    return flce.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flce_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_exported_set(lib):
    declared = _declared_functions()
    assert declared == sorted(B.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name


def test_version_and_strerror(lib):
    assert lib.flce_version() == 300
    for code in range(0, 10):
        assert lib.flce_strerror(code)
        assert b"unknown" not in lib.flce_strerror(code)
    assert b"unknown" in lib.flce_strerror(99)


def test_error_codes_match_the_header():
    """Every FLCE_ERR_* code of the header has its name in the binding's error messages."""
    codes = dict((name, int(v)) for name, v in
                 re.findall(r"FLCE_ERR_([A-Z_]+)\s*=\s*(\d+)", open(HEADER).read()))
    assert codes and max(codes.values()) == 10
    assert {v: k for k, v in codes.items()} == B._ERR_NAMES


def test_params_struct_layout():
    # int64 x4, int32, float, float, int32, int64, int32, float, pointer, int64 x3, int32
    # (+ 4 bytes of tail padding) -> 104 bytes, as in flce.h
    assert ctypes.sizeof(B.FlceParams) == 104
    assert B.FlceParams.chunk_v.offset == 48
    assert B.FlceParams.weight_layout.offset == 56
    assert B.FlceParams.label_smoothing.offset == 60
    assert B.FlceParams.class_weight.offset == 64
    assert B.FlceParams.v_offset.offset == 72
    assert B.FlceParams.v_total.offset == 80
    assert B.FlceParams.chunk_n.offset == 88
    assert B.FlceParams.dhidden_fp32.offset == 96


def test_params_struct_matches_the_c_compiler(tmp_path):
    """sizeof / offsetof of flce_params from the C compiler agree with the binding."""
    import subprocess
    src = tmp_path / "t.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "flce.h"\n'
        'int main(void){printf("%zu %zu %zu %zu %zu %zu %zu\\n", sizeof(flce_params),'
        ' offsetof(flce_params, chunk_v), offsetof(flce_params, class_weight),'
        ' offsetof(flce_params, v_offset), offsetof(flce_params, v_total),'
        ' offsetof(flce_params, chunk_n), offsetof(flce_params, dhidden_fp32)); return 0;}\n')
    exe = tmp_path / "t"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    F = B.FlceParams
    assert [int(x) for x in out] == [ctypes.sizeof(F), F.chunk_v.offset, F.class_weight.offset,
                                     F.v_offset.offset, F.v_total.offset, F.chunk_n.offset,
                                     F.dhidden_fp32.offset]


def test_workspace_sizes(lib):
    p = flce.make_params(8192, 4096, 128256, "mean", zloss_coef=1e-4)
    fwd = flce.workspace_size(p, 0)
    # (m, d, s) partials: at least one part per 256-column tile, per row
    n_parts = (128256 + 255) // 256
    assert fwd >= 3 * n_parts * 8192 * 4 + 3 * 8192 * 4
    bwd = flce.workspace_size(p, 1)
    assert bwd >= 8192 * 16  # per-row constants
    # an explicit chunk width: dlogits chunk N*Vc*2 plus an fp32 dhidden accumulator
    p2 = flce.make_params(300, 200, 1000, "none", chunk_v=256)
    assert flce.workspace_size(p2, 1) >= 300 * 256 * 2 + 300 * 200 * 4
    assert flce.kernel_launches(p2, 1) == 1 + 3 * 4
    assert flce.kernel_launches(p2, 0) == 2
    assert flce.kernel_launches(flce.make_params(300, 200, 1000, "sum"), 0) == 3
    # an fp32 dhidden is its own accumulator: no fp32 workspace copy of it
    p3 = flce.make_params(300, 200, 1000, "none", chunk_v=256, dhidden_fp32=True)
    assert flce.workspace_size(p3, 1) == flce.workspace_size(p2, 1) - ((300 * 200 * 4 + 255)
                                                                       // 256 * 256)


def test_fused_workspace_and_launches(lib):
    # gradient in forward: fp32 logits + bf16 dlogits of one token chunk (auto: the
    # Llama-3 head shape fits one chunk), no dweight accumulator for a single chunk
    p = flce.make_params(8192, 4096, 128256, "mean", zloss_coef=1e-4)
    ws = flce.workspace_size(p, 3)
    assert 8192 * 128256 * 6 <= ws < 8192 * 128256 * 6 + (256 << 20)
    assert flce.kernel_launches(p, 4) == 6 + 1
    # explicit chunks of 512 rows: 3 chunks for 1100 rows, plus an fp32 dweight accumulator
    p2 = flce.make_params(1100, 64, 1000, "none", chunk_n=512)
    assert flce.workspace_size(p2, 3) >= 512 * 1024 * 6 + 64 * 1000 * 4
    assert flce.kernel_launches(p2, 4) == 6 * 3
    # one chunk when N fits: no accumulator
    p3 = flce.make_params(300, 64, 1000, "sum", chunk_n=512)
    assert flce.workspace_size(p3, 3) < 512 * 1024 * 6 + 64 * 1000 * 4
    assert flce.kernel_launches(p3, 4) == 6 + 1


@pytest.mark.parametrize("kw,code", [
    (dict(N=10, H=7 * 8 + 4, V=64), 3),     # H % 8
    (dict(N=10, H=64, V=100), 3),           # V % 8
    (dict(N=10, H=4, V=64), 2),             # H < 8
    (dict(N=-1, H=64, V=64), 2),
    (dict(N=10, H=64, V=0), 2),
    (dict(N=10, H=64, V=64, chunk_v=100), 1),
    (dict(N=10, H=64, V=64, chunk_n=256), 1),               # chunk_n % 512
    (dict(N=10, H=64, V=64, zloss_coef=-1.0), 1),
    (dict(N=10, H=64, V=64, weight_layout=7), 1),
    (dict(N=10, H=64, V=64, label_smoothing=1.5), 1),
    (dict(N=10, H=64, V=64, label_smoothing=-0.1), 1),
    (dict(N=10, H=64, V=64, v_offset=8), 1),                  # offset without a total
    (dict(N=10, H=64, V=64, v_offset=8, v_total=64), 2),      # shard past the vocabulary
    (dict(N=10, H=64, V=64, v_total=128, label_smoothing=0.1), 1),
])
def test_bad_params_rejected_on_host(lib, kw, code):
    args = dict(N=10, H=64, V=64)
    args.update(kw)
    red = args.pop("reduction", "mean")
    bad_layout = args.pop("weight_layout", None)
    p = flce.make_params(args.pop("N"), args.pop("H"), args.pop("V"), red, **args)
    if bad_layout is not None:
        p.weight_layout = bad_layout
    assert lib.flce_workspace_size(ctypes.byref(p), 0) == 0
    fake = ctypes.c_void_p(0x1000)
    rc = lib.flce_forward(ctypes.byref(p), fake, fake, fake, fake, fake, fake, fake, fake,
                          1 << 20, None)
    assert rc == code
    rc = lib.flce_backward(ctypes.byref(p), fake, fake, fake, fake, fake, fake, fake, fake,
                           fake, fake, 1 << 20, None)
    assert rc == code
    assert lib.flce_workspace_size(ctypes.byref(p), 3) == 0
    rc = lib.flce_forward_backward(ctypes.byref(p), fake, fake, fake, fake, fake, fake, fake,
                                   fake, fake, fake, fake, fake, 1 << 20, None)
    assert rc == code


def test_fused_rejects_shards_nulls_alignment_and_small_workspace(lib):
    ok = ctypes.c_void_p(0x10000)
    bad = ctypes.c_void_p(0x10004)
    # a partial vocabulary shard has no whole-vocabulary logsumexp to form dlogits with
    p = flce.make_params(10, 64, 64, "mean", v_offset=64, v_total=128)
    args = [ok] * 12
    assert lib.flce_forward_backward(ctypes.byref(p), *args, 1 << 20, None) == 1
    p = flce.make_params(10, 64, 64, "mean")
    nulls = list(args)
    nulls[9] = None  # dhidden
    assert lib.flce_forward_backward(ctypes.byref(p), *nulls, 1 << 20, None) == 1
    mis = list(args)
    mis[10] = bad  # dweight
    assert lib.flce_forward_backward(ctypes.byref(p), *mis, 1 << 20, None) == 3
    assert lib.flce_forward_backward(ctypes.byref(p), *args, 16, None) == 4


def test_vocabulary_alignment_applies_to_the_hv_layout_only(lib):
    """V is a row length only in the [H,V] layout; a [V,H] weight takes any V."""
    for V in (1, 7, 1001, 50257):
        p = flce.make_params(10, 64, V, "mean", weight_layout="vh")
        for phase in (0, 1, 3):
            assert lib.flce_workspace_size(ctypes.byref(p), phase) > 0
        q = flce.make_params(10, 64, V, "mean", weight_layout="hv")
        assert lib.flce_workspace_size(ctypes.byref(q), 0) == 0
        fake = ctypes.c_void_p(0x1000)
        assert lib.flce_forward(ctypes.byref(q), fake, fake, fake, fake, fake, fake, fake, fake,
                                1 << 20, None) == 3
    # H is a row length in both layouts
    p = flce.make_params(10, 60, 64, "mean", weight_layout="vh")
    assert lib.flce_workspace_size(ctypes.byref(p), 0) == 0


def test_check_params_gives_the_entry_points_status(lib):
    """flce_check_params returns the status the entry points return for the same
    parameters, and the binding raises it (not a generic BAD_ARG) when sizing."""
    cases = [(dict(N=10, H=64, V=100), 3), (dict(N=10, H=4, V=64), 2),
             (dict(N=10, H=64, V=64, chunk_v=100), 1), (dict(N=10, H=64, V=100,
                                                             weight_layout="vh"), 0)]
    for kw, code in cases:
        p = flce.make_params(kw.pop("N"), kw.pop("H"), kw.pop("V"), "mean", **kw)
        assert lib.flce_check_params(ctypes.byref(p)) == code
        if code:
            with pytest.raises(B.FlceError) as ei:
                flce.workspace_size(p, 0)
            assert ei.value.code == code
    assert lib.flce_check_params(None) == 1


def test_fp32_dhidden_needs_32_byte_alignment_and_a_flag_of_0_or_1(lib):
    ok = ctypes.c_void_p(0x10000)
    half = ctypes.c_void_p(0x10010)  # 16-byte aligned, not 32
    p = flce.make_params(10, 64, 64, "mean", dhidden_fp32=True)
    args = [ok] * 7 + [half, ok, ok]  # dhidden is the 8th pointer
    assert lib.flce_backward(ctypes.byref(p), *args, 1 << 20, None) == 3
    p16 = flce.make_params(10, 64, 64, "mean")  # a bf16 dhidden may sit there
    assert lib.flce_backward(ctypes.byref(p16), *args, 16, None) == 4  # gets past alignment
    p.dhidden_fp32 = 2
    assert lib.flce_workspace_size(ctypes.byref(p), 1) == 0
    assert lib.flce_backward(ctypes.byref(p), *([ok] * 10), 1 << 20, None) == 1


def test_scale_bf16_argument_checks(lib):
    ok = ctypes.c_void_p(0x10000)
    assert lib.flce_scale_bf16(ok, -1, ok, None) == 1
    assert lib.flce_scale_bf16(ok, 8, None, None) == 1
    assert lib.flce_scale_bf16(None, 8, ok, None) == 1
    assert lib.flce_scale_bf16(ctypes.c_void_p(0x10002), 8, ok, None) == 3
    assert lib.flce_scale_bf16(ok, 0, ok, None) == 0


def test_bad_reduction_and_nulls(lib):
    p = flce.make_params(10, 64, 64, "mean")
    p.reduction = 7
    assert lib.flce_forward(ctypes.byref(p), None, None, None, None, None, None, None, None,
                            0, None) == 1
    p = flce.make_params(10, 64, 64, "mean")
    assert lib.flce_forward(ctypes.byref(p), None, None, None, None, None, None, None, None,
                            0, None) == 1
    assert lib.flce_forward(None, None, None, None, None, None, None, None, None, 0, None) == 1


def test_misaligned_pointer_and_small_workspace(lib):
    p = flce.make_params(10, 64, 64, "mean")
    ok = ctypes.c_void_p(0x10000)
    bad = ctypes.c_void_p(0x10004)
    rc = lib.flce_forward(ctypes.byref(p), bad, ok, ok, ok, ok, ok, ok, ok, 1 << 20, None)
    assert rc == 3
    rc = lib.flce_forward(ctypes.byref(p), ok, ok, ok, ok, ok, ok, ok, ok, 16, None)
    assert rc == 4


def test_product_path_fails_loudly_without_library(tmp_path):
    saved = B._lib
    B._lib = None
    try:
        with pytest.raises(RuntimeError, match="missing"):
            B.load_library(str(tmp_path / "nope.so"))
    finally:
        B._lib = saved


def test_cpu_tensors_are_refused_not_computed():
    """There is no CPU fallback: host tensors are refused before anything runs."""
    import torch
    h = torch.zeros(16, 64, dtype=torch.bfloat16)
    w = torch.zeros(64, 128, dtype=torch.bfloat16)
    y = torch.zeros(16, dtype=torch.int64)
    g = torch.ones(1)
    calls = [
        lambda: flce.flce_forward(h, w, y, "mean"),
        lambda: flce.flce_backward(h, w, y, torch.zeros(16), torch.zeros(16), g, g, "mean"),
        lambda: flce.flce_forward_backward(h, w, y, g, g, "mean"),
        lambda: flce.linear_cross_entropy(h, w, y, "mean"),
        lambda: flce.linear_cross_entropy(h, w, y, "mean", grad_in_forward=True),
        lambda: flce.flce_shard_stats(h, w, y, 0, 128),
        lambda: flce.flce_scale_bf16(h, g),
    ]
    for call in calls:
        with pytest.raises(TypeError, match="CUDA"):
            call()


def test_selftest_wait_timeout_argument_checks(lib):
    ok = ctypes.c_void_p(0x10000)
    assert lib.flce_selftest_wait_timeout(None, 256, 1000, None) == 1
    assert lib.flce_selftest_wait_timeout(ctypes.c_void_p(0x10010), 256, 1000, None) == 3
    assert lib.flce_selftest_wait_timeout(ok, 256, 0, None) == 1
    assert lib.flce_selftest_wait_timeout(ok, 256, 3_000_000_000, None) == 1
    assert lib.flce_selftest_wait_timeout(ok, 16, 1000, None) == 4


def test_plain_c_program_links_and_calls_the_library(lib, tmp_path):
    """The boundary is a C ABI: a C program (no Python, no torch) links libflce.so, sizes
    a workspace and gets the documented host-side errors back (no GPU needed)."""
    import subprocess
    src = tmp_path / "use_flce.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "flce.h"
int main(void) {
  flce_params p;
  memset(&p, 0, sizeof(p));
  p.N = 8192; p.H = 4096; p.V = 128256; p.ignore_index = -100;
  p.reduction = FLCE_RED_MEAN; p.zloss_coef = 1e-4f;
  size_t ws0 = flce_workspace_size(&p, 0), ws1 = flce_workspace_size(&p, 1);
  int bad_null = flce_forward(&p, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL);
  p.H = 4100;  /* not a multiple of 8 */
  int bad_align = flce_forward(&p, (void*)0x1000, (void*)0x1000, (void*)0x1000, (void*)0x1000,
                               (void*)0x1000, (void*)0x1000, (void*)0x1000, (void*)0x1000,
                               1 << 20, NULL);
  printf("%d %zu %zu %d %d %s\n", flce_version(), ws0, ws1, bad_null, bad_align,
         flce_strerror(FLCE_ERR_ALIGN));
  return 0;
}
''')
    exe = tmp_path / "use_flce"
    libdir = os.path.dirname(B.LIB_PATH)
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-L", libdir,
                    "-l:libflce.so", "-Wl,-rpath," + libdir, "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    p = flce.make_params(8192, 4096, 128256, "mean", zloss_coef=1e-4)
    assert int(out[0]) == lib.flce_version()
    assert int(out[1]) == flce.workspace_size(p, 0)
    assert int(out[2]) == flce.workspace_size(p, 1)
    assert int(out[3]) == 1 and int(out[4]) == 3
    assert "aligned" in " ".join(out[5:])


def test_auto_chunking_follows_the_documented_rules(lib):
    """flce.h: the backward's chunk_v = 0 picks the widest multiple of 256 columns whose bf16
    dlogits [N, chunk_v] fit 2 GiB; flce_forward_backward's chunk_n = 0 the largest multiple
    of 512 rows whose fp32 logits and bf16 dlogits (V rounded up to 256) fit 8 GiB.  Checked
    through the launch counts (3 GEMMs per vocabulary chunk, 6 launches per token chunk)."""
    import random
    rng = random.Random(5)
    cdiv = lambda a, b: -(-a // b)  # noqa: E731
    for _ in range(200):
        N = rng.choice([1, 7, 300, 4096, 8192, 16384, 65536, 200000])
        V = 8 * rng.randint(1, 40000)
        vc = max(256, min((2 << 30) // (2 * N) // 256 * 256, cdiv(V, 256) * 256))
        p = flce.make_params(N, 64, V, "none")
        assert flce.kernel_launches(p, 1) == 1 + 3 * cdiv(V, vc), (N, V)
        ldz = cdiv(V, 256) * 256
        nc = max(512, (8 << 30) // (ldz * 6) // 512 * 512)
        nc = min(nc, cdiv(N, 256) * 256)
        assert flce.kernel_launches(p, 4) == 6 * cdiv(N, nc), (N, V)


def test_random_parameter_sets_follow_the_documented_rules(lib):
    """Seeded fuzz of flce_check_params / flce_workspace_size against the rules flce.h
    states: random valid parameter sets pass and get a workspace for every phase; the
    same sets with exactly one documented rule broken get that rule's status and no
    workspace."""
    import random
    r = random.Random(2024)
    OK, BAD_ARG, BAD_SHAPE, ALIGN = 0, 1, 2, 3

    def valid():
        layout = r.choice(["hv", "vh"])
        V = r.choice([1, 7, 8, 255, 256, 1000, 50257, 128256, 1 << 20])
        if layout == "hv":
            V = max(8, V // 8 * 8)
        kw = dict(N=r.choice([0, 1, 300, 8192, 1 << 20]), H=8 * r.randint(1, 1024), V=V,
                  reduction=r.choice(["none", "mean", "sum"]),
                  zloss_coef=r.choice([0.0, 1e-4]), softcap=r.choice([0.0, 30.0]),
                  chunk_v=r.choice([0, 256, 65536]), weight_layout=layout,
                  chunk_n=r.choice([0, 512, 8192]), dhidden_fp32=r.random() < 0.3)
        if r.random() < 0.3:  # a vocabulary shard
            kw["v_total"] = V + r.choice([0, 8, 1000])
            kw["v_offset"] = r.randint(0, kw["v_total"] - V)
        elif r.random() < 0.3:
            kw["label_smoothing"] = r.choice([0.0, 0.1, 1.0])
        return kw

    breakers = [  # (rule of flce.h, how to break it, status)
        ("H >= 8", lambda k: k.update(H=0), BAD_SHAPE),
        ("V >= 1", lambda k: k.update(V=0), BAD_SHAPE),
        ("N >= 0", lambda k: k.update(N=-5), BAD_SHAPE),
        ("H % 8 == 0", lambda k: k.update(H=k["H"] + 4), ALIGN),
        ("V % 8 == 0 for [H,V]", lambda k: k.update(weight_layout="hv", V=8 * (k["V"] // 8 + 1) + 3,
                                                   v_total=0, v_offset=0), ALIGN),
        ("chunk_v a multiple of 256", lambda k: k.update(chunk_v=300), BAD_ARG),
        ("chunk_n a multiple of 512", lambda k: k.update(chunk_n=1000), BAD_ARG),
        ("zloss_coef >= 0", lambda k: k.update(zloss_coef=-1.0), BAD_ARG),
        ("softcap >= 0", lambda k: k.update(softcap=-2.0), BAD_ARG),
        ("label_smoothing in [0, 1]", lambda k: k.update(label_smoothing=1.5, v_total=0,
                                                          v_offset=0), BAD_ARG),
        ("v_offset only with v_total", lambda k: k.update(v_total=0, v_offset=8), BAD_ARG),
        ("shard inside the vocabulary", lambda k: k.update(v_total=k["V"], v_offset=8,
                                                            label_smoothing=0.0), BAD_SHAPE),
        ("no smoothing with shards", lambda k: k.update(v_total=k["V"] + 8, v_offset=0,
                                                        label_smoothing=0.1), BAD_ARG),
    ]
    seen = set()
    for _ in range(400):
        kw = valid()
        rule, expect = None, OK
        if r.random() < 0.6:
            rule, brk, expect = r.choice(breakers)
            brk(kw)
            seen.add(rule)
        args = dict(kw)
        p = flce.make_params(args.pop("N"), args.pop("H"), args.pop("V"),
                             args.pop("reduction"), **args)
        assert lib.flce_check_params(ctypes.byref(p)) == expect, (rule, kw)
        for phase in (0, 1, 2):
            n = lib.flce_workspace_size(ctypes.byref(p), phase)
            assert (n > 0) == (expect == OK), (rule, kw, phase)
    assert seen == {b[0] for b in breakers}
