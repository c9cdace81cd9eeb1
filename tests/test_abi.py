"""The C-ABI library loads and exports every function include/dpp.h declares;
host-side argument checks (no GPU needed: they fail before any CUDA call)."""
import ctypes
import os
import re

import pytest
import torch

import stale_activations_gb300 as dpp
from stale_activations_gb300 import build as dbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    dbuild.build_library()
    return dpp.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "dpp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_four_calls():
    names = _declared_functions()
    for n in ("patch_layer_step", "halo_conv3x3", "stale_kv_attention", "refresh_residual"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"libdpp.so does not export {n}"
    assert set(dpp.EXPORTS) <= set(names)


def test_plain_c_consumer_compiles_links_and_agrees_on_layouts(lib, tmp_path):
    """tests/abi_check.c, plain C99 against include/dpp.h, linked with libdpp.so: host
    checks from C, and the struct sizes C sees equal the binding's."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "abi_check"
    libdir = os.path.dirname(dbuild.LIB)
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "abi_check.c"), "-o", str(exe), "-L", libdir,
                    "-ldpp", f"-Wl,-rpath,{libdir}"], check=True)
    env = dict(os.environ)
    env["LD_LIBRARY_PATH"] = libdir + os.pathsep + env.get("LD_LIBRARY_PATH", "")
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, env=env).stdout
    sizes = [int(v) for v in out.split("sizes")[1].split()]
    assert sizes == [ctypes.sizeof(dpp.LayerParams), ctypes.sizeof(dpp.LayerWeights),
                     ctypes.sizeof(dpp.LayerState), ctypes.sizeof(dpp.WorkspaceLayout)]


def test_status_strings(lib):
    assert dpp.status_string(0) == "ok"
    assert "timeout" in dpp.status_string(6)
    assert lib.dpp_version() >= 100


def _params(**kw):
    raw = kw.pop("fuse_gn_raw", None)   # a value make_params would not produce
    base = dict(B=2, H=64, W=64, C=640, P=4, G=32, heads=10, dtype=dpp.BF16)
    base.update(kw)
    prm = dpp.make_params(**base)
    if raw is not None:
        prm.fuse_gn = raw
    return prm


def test_workspace_layout_sizes(lib):
    prm = _params()
    lo = dpp.workspace_layout(prm)
    act = 2 * 64 * 64 * 640 * 2
    assert lo.total >= 6 * act
    offs = [lo.status, lo.gn_partial, lo.gn_fresh, lo.gn_params, lo.y, lo.h, lo.q, lo.k, lo.v, lo.o,
            lo.attn_partial]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert lo.y == lo.gn_params                          # no parameters without fuse_gn
    lf = dpp.workspace_layout(_params(fuse_gn=1))
    assert lf.y - lf.gn_params >= 2 * 4 * 3 * 640 * 4   # [B, P, 3, C] fp32 parameters
    # the maxima of |V| per (batch, head) (20 words, 256 bytes with padding); then 320
    # attention units on (without a GPU, the library assumes) 152 SMs: one round of 152
    # whole units, the other 168 shared; a counter per shared unit, query tile and 32-row
    # warp (8 x 168 words = 5376 bytes), then 152 + 168 partial records of 34816 bytes
    part = dpp.attention_scratch_size(2, 4096, 10, 4, split=True)
    assert part == 256 + 5376 + (152 + 168) * 34816 or torch.cuda.is_available()
    assert dpp.attention_scratch_size(2, 4096, 10, 4, split=False) == 256
    assert dpp.attention_scratch_size(2, 4096, 10, 4, dtype=dpp.F32) == 0
    assert lo.attn_partial_bytes == part and lo.total >= lo.attn_partial + part
    n, nb = dpp.message_sizes(prm)
    blc = 2 * 4096 * 640
    assert n == 2 * blc + 2 * 3 * 2 * 64 * 640
    assert nb == 2 * blc // 128 + 2 * 3 * (2 * 64 * 640 // 128)


@pytest.mark.parametrize("kw", [dict(H=63), dict(P=3), dict(C=600, heads=10), dict(G=7),
                                dict(heads=5), dict(dtype=7), dict(W=44), dict(W=48, fuse_gn=1),
                                dict(gn_mode=3),
                                dict(gn_mode=-1), dict(fuse_gn_raw=2),
                                dict(dtype=dpp.F32, fuse_refresh=1),
                                dict(B=1, H=32, W=32, C=64, P=2, G=8, heads=1, dtype=dpp.F32,
                                     fuse_gn=1)])
def test_invalid_params_rejected(lib, kw):
    prm = _params(**kw)
    assert lib.dpp_workspace_size(ctypes.byref(prm)) == 0
    lo = dpp.WorkspaceLayout()
    assert lib.dpp_workspace_query(ctypes.byref(prm), ctypes.byref(lo)) != 0


def test_fp32_tiny_params_accepted(lib):
    prm = _params(B=1, H=32, W=32, C=64, P=2, G=8, heads=1, dtype=dpp.F32)
    assert dpp.workspace_size(prm) > 0
    assert dpp.layer_kernel_count(prm, dpp.SYNC) == 6
    assert dpp.layer_kernel_count(prm, dpp.STALE) == 7


def test_host_checks_without_launch(lib):
    vp = ctypes.c_void_p
    # n == 0 is a no-op, null pointers / bad dtype / bad sizes are rejected
    assert lib.refresh_residual(None, None, None, None, 0, dpp.BF16, None) == 0
    assert lib.refresh_residual(None, None, None, None, 5, dpp.BF16, None) == 1
    assert lib.refresh_residual(vp(16), vp(16), vp(16), vp(16), 5, 9, None) == 4
    assert lib.refresh_residual(vp(16), vp(16), vp(16), vp(16), -1, dpp.BF16, None) == 2
    assert lib.refresh_residual(vp(16), vp(24), vp(16), vp(16), 5, dpp.BF16, None) == 3
    # the receiver's half: same argument rules
    assert lib.apply_residual(None, None, None, 0, dpp.BF16, None) == 0
    assert lib.apply_residual(None, vp(16), vp(16), 5, dpp.BF16, None) == 1
    assert lib.apply_residual(vp(16), vp(16), vp(16), 5, 9, None) == 4
    assert lib.apply_residual(vp(16), vp(16), vp(24), 5, dpp.BF16, None) == 3
    assert lib.apply_residual(vp(16), vp(18), vp(16), 5, dpp.BF16, None) == 3
    assert lib.halo_conv3x3(None, None, None, None, 1, 8, 8, 64, 128, 2, dpp.BF16, None, None) == 1
    a = vp(256)
    assert lib.halo_conv3x3(a, a, a, a, 1, 9, 64, 64, 128, 2, dpp.BF16, None, None) == 2
    assert lib.halo_conv3x3(a, a, a, a, 1, 8, 64, 64, 100, 2, dpp.BF16, None, None) == 2
    # bf16: W a multiple of 8 and H*W a multiple of 128 (row segments of gcd(W, 128))
    assert lib.halo_conv3x3(a, a, a, a, 1, 16, 44, 64, 128, 2, dpp.BF16, None, None) == 2
    assert lib.halo_conv3x3(a, a, a, a, 1, 3, 40, 64, 128, 3, dpp.BF16, None, None) == 2
    assert lib.stale_kv_attention(a, a, a, a, a, a, 1, 1024, 2, 32, 2, dpp.BF16, a, 4096, None,
                                  None) == 2
    assert lib.stale_kv_attention(a, a, a, a, a, a, 1, 1000, 2, 64, 3, dpp.BF16, a, 4096, None,
                                  None) == 2
    assert lib.stale_kv_attention(a, a, a, a, a, vp(8), 1, 1024, 2, 64, 2, dpp.BF16, a, 4096,
                                  None, None) == 3
    # a missing or short scratch buffer is refused before any launch, for both schedules
    for fn, split in ((lib.stale_kv_attention, 0), (lib.stale_kv_attention_split, 1)):
        need = lib.dpp_attention_scratch_size(1, 1024, 2, 64, 4, dpp.BF16, split)
        assert need > 0
        assert fn(a, a, a, a, a, a, 1, 1024, 2, 64, 4, dpp.BF16, None, 0, None, None) == 9
        assert fn(a, a, a, a, a, a, 1, 1024, 2, 64, 4, dpp.BF16, a, need - 1, None, None) == 9
        assert fn(a, a, a, a, a, a, 1, 1024, 2, 64, 4, dpp.BF16, vp(264), need, None, None) == 3
    assert lib.dpp_attention_scratch_size(1, 1000, 2, 64, 3, dpp.BF16, 1) == 0  # invalid shape
    prm = _params()
    w = dpp.LayerWeights()
    st = dpp.LayerState()
    assert lib.patch_layer_step(ctypes.byref(prm), ctypes.byref(w), ctypes.byref(st), a, a, 0, a,
                                None) == 1
    # the second state set: all four or none (1), none equal to its counterpart (9), the
    # same alignment rules (3) -- all refused before any launch
    w = dpp.LayerWeights(*[vp(256 * (i + 1)) for i in range(5)])
    cur = [vp(0x10000 * (i + 1)) for i in range(6)]
    nxt = [vp(0x100000 * (i + 1)) for i in range(4)]
    for bad, code in ((nxt[:3] + [None], 1), ([cur[0]] + nxt[1:], 9), (nxt[:1] + [vp(0x200008)] + nxt[2:], 3)):
        st = dpp.LayerState(*cur, *bad)
        assert lib.patch_layer_step(ctypes.byref(prm), ctypes.byref(w), ctypes.byref(st), a, a,
                                    dpp.STALE, a, None) == code, bad


def test_otil_host_checks(lib):
    ok = dpp.otil_params(2, 4, 128, 128, 4, 8, 32, 4)
    assert dpp.otil_blocks(ok) == (32 // 8) * (128 // 32)
    for kw in (dict(P=1), dict(H=130), dict(bh=5), dict(bw=48), dict(k=0), dict(k=17),
               dict(dtype=7)):
        base = dict(B=2, C=4, H=128, W=128, P=4, bh=8, bw=32, k=4, dtype=dpp.BF16)
        base.update(kw)
        bad = dpp.otil_params(**base)
        assert dpp.otil_blocks(bad) == -1
        assert lib.dpp_otil_step(ctypes.byref(bad), None, None, None, None, None, None) != 0
    a = ctypes.c_void_p(256)
    assert lib.dpp_otil_step(ctypes.byref(ok), None, a, a, a, a, None) == 1
    assert lib.dpp_otil_step(ctypes.byref(ok), ctypes.c_void_p(257), a, a, a, a, None) == 3
