"""The C-ABI library: it builds, loads, exports every symbol include/pkv.h
declares, and rejects bad arguments on the host before touching a device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(pkv_\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    from paged_kv_attention_05_gb300 import build as b
    b.build()
    import paged_kv_attention_05_gb300 as pkv
    return pkv.load()


def test_header_declares_the_two_calls_and_helpers():
    names = _declared()
    for n in ["pkv_write", "pkv_attention", "pkv_reserve_workspace", "pkv_get_error",
              "pkv_last_error_string", "pkv_num_sms"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import paged_kv_attention_05_gb300 as pkv
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)$", out, flags=re.M))
    for n in _declared():
        assert n in exported, n
        assert hasattr(lib, n)


def test_header_compiles_as_plain_c():
    src = '#include "pkv.h"\nint main(void){return PKV_OK;}\n'
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-x", "c", "-", "-o", "/dev/null"], input=src, text=True,
                       capture_output=True)
    assert r.returncode == 0, r.stderr


FAKE = 0x10000  # a non-null, 16-byte aligned address; never dereferenced by these calls


def test_write_rejects_bad_geometry_on_host(lib):
    # block_size 8: unsupported, returned before any CUDA call
    rc = lib.pkv_write(FAKE, 1024, FAKE, 1024, FAKE, FAKE, 10, 8, 8, 128, FAKE, 4, None)
    assert rc == -2
    assert b"block_size" in lib.pkv_last_error_string()
    rc = lib.pkv_write(FAKE, 1024, FAKE, 1024, FAKE, FAKE, 10, 16, 8, 64, FAKE, 4, None)
    assert rc == -2
    rc = lib.pkv_write(FAKE, 1024, FAKE, 1024, FAKE, FAKE, 10, 16, 8, 128, FAKE, -1, None)
    assert rc == -1
    rc = lib.pkv_write(FAKE, 1000, FAKE, 1024, FAKE, FAKE, 10, 16, 8, 128, FAKE, 4, None)
    assert rc == -1   # row stride below Hkv * 128
    rc = lib.pkv_write(FAKE + 2, 1024, FAKE, 1024, FAKE, FAKE, 10, 16, 8, 128, FAKE, 4, None)
    assert rc == -3   # misaligned
    rc = lib.pkv_write(None, 1024, FAKE, 1024, FAKE, FAKE, 10, 16, 8, 128, FAKE, 4, None)
    assert rc == -1
    # nothing to do is not an error
    assert lib.pkv_write(None, 0, None, 0, None, None, 10, 16, 8, 128, None, 0, None) == 0


def test_attention_rejects_bad_geometry_on_host(lib):
    args = dict(q=FAKE, qs=4096, rows=4, hq=32, kc=FAKE, vc=FAKE, nb=10, bs=16, hkv=8, d=128,
                qsl=FAKE, sl=FAKE, bt=FAKE, w=4, R=2, scale=0.088, out=FAKE, os=4096)

    def call(**kw):
        a = dict(args, **kw)
        return lib.pkv_attention(a["q"], a["qs"], a["rows"], a["hq"], a["kc"], a["vc"], a["nb"],
                                 a["bs"], a["hkv"], a["d"], a["qsl"], a["sl"], a["bt"], a["w"],
                                 a["R"], a["scale"], a["out"], a["os"], None)

    assert call(hq=30) == -2                  # Hq not a multiple of Hkv
    assert call(hq=64 * 8, qs=64 * 8 * 128, os=64 * 8 * 128) == -2   # G = 64 > 32
    assert call(bs=32) == -2
    assert call(d=256) == -2
    assert call(R=-1) == -1
    assert call(qs=100) == -1
    assert call(out=FAKE + 8) == -3
    assert call(qsl=None) == -1
    assert call(scale=float("nan")) == -1
    assert call(R=0) == 0 and call(rows=0) == 0


def test_python_binding_requires_cuda_tensors():
    torch = pytest.importorskip("torch")
    import paged_kv_attention_05_gb300 as pkv
    k = torch.zeros(2, 8, 128, dtype=torch.bfloat16)
    kc = torch.zeros(4, 16, 8, 128, dtype=torch.bfloat16)
    sm = torch.zeros(2, dtype=torch.int64)
    with pytest.raises(ValueError):
        pkv.pkv_write(k, k, kc, kc, sm)
    with pytest.raises(TypeError):
        pkv.pkv_write(k.float(), k, kc, kc, sm)


def test_int8_and_plan_calls_reject_bad_arguments_on_host(lib):
    ct = ctypes
    i64, i32, f32, vp = ct.c_int64, ct.c_int32, ct.c_float, ct.c_void_p
    lib.pkv_write_int8.restype = ct.c_int
    lib.pkv_write_int8.argtypes = [vp, i64, vp, i64, vp, vp, f32, f32, i64, i32, i32, i32, vp, i64,
                                   vp]
    lib.pkv_attention_int8.restype = ct.c_int
    lib.pkv_attention_int8.argtypes = [vp, i64, i64, i32, vp, vp, f32, f32, i64, i32, i32, i32,
                                       vp, vp, vp, i64, i32, f32, vp, i64, vp]
    lib.pkv_plan.restype = ct.c_int
    lib.pkv_plan.argtypes = [i64, i32, i32, vp, vp, i64, i32, vp]
    lib.pkv_attention_planned.restype = ct.c_int
    lib.pkv_attention_planned.argtypes = [vp, i64, i32, vp, vp, i64, i32, i32, i32, vp, f32, vp,
                                          i64, vp]
    # int8 write: scales must be finite and positive; geometry as pkv_write
    w8 = lambda ks, vs, bs=16: lib.pkv_write_int8(FAKE, 1024, FAKE, 1024, FAKE, FAKE, ks, vs, 10,
                                                  bs, 8, 128, FAKE, 4, None)
    assert w8(0.0, 0.1) == -1 and w8(0.1, float("nan")) == -1 and w8(-1.0, 0.1) == -1
    assert w8(float("inf"), 0.1) == -1 and w8(0.1, 0.1, bs=8) == -2
    # int8 attention: the same checks as pkv_attention, plus the scales
    a8 = lambda ks, vs, hq=32: lib.pkv_attention_int8(FAKE, 4096, 4, hq, FAKE, FAKE, ks, vs, 10,
                                                      16, 8, 128, FAKE, FAKE, FAKE, 4, 2, 0.088,
                                                      FAKE, 4096, None)
    assert a8(0.0, 0.1) == -1 and a8(0.1, 0.1, hq=30) == -2
    # the plan: metadata checks of pkv_attention
    pl = lambda hq=32, hkv=8, w=4, R=2, qsl=FAKE: lib.pkv_plan(4, hq, hkv, qsl, FAKE, w, R, None)
    assert pl(hq=30) == -2 and pl(hkv=0) == -1 and pl(R=-1) == -1 and pl(qsl=None) == -1
    assert pl(w=40000) == -2
    # a planned call: geometry checked before the device is looked at
    ap = lambda bs=16, d=128, hkv=8: lib.pkv_attention_planned(FAKE, 4096, 32, FAKE, FAKE, 10, bs,
                                                               hkv, d, FAKE, 0.088, FAKE, 4096,
                                                               None)
    assert ap(bs=32) == -2 and ap(d=64) == -2 and ap(hkv=40000) == -2
