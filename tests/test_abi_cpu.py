"""The C ABI library on a machine without a GPU: it loads, exports every declared entry
point, and rejects bad arguments before touching the device (no compute calls here)."""

import ctypes
import re
from pathlib import Path

import pytest

from paged_kv_cache_244_gb300 import _build

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def L():
    from paged_kv_cache_244_gb300 import binding
    _build.build()
    return binding.lib()


def declared_functions():
    names = []
    for header in sorted((ROOT / "include").glob("*.h")):
        text = re.sub(r"/\*.*?\*/", "", header.read_text(), flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w ]*?\**\s*\**(pa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("pa_rope_kv_store", "pa_decode", "pa_decode_workspace_size",
                 "pa_decode_partition_tokens", "pa_get_device_status", "pa_status_string",
                 "pa_selftest_wait_timeout", "pa_decode_static_workspace", "pa_decode_step",
                 "pa_copy_blocks", "pa_rope_kv_store_fp8", "pa_decode_fp8", "pa_decode_step_fp8",
                 "pa_prefill", "pa_gather_checksum", "pa_gather_checksum_fp8", "pa_stage_copy",
                 "pa_set_timing_jitter"):
        assert must in names


def test_header_is_plain_c_and_links(L, tmp_path):
    """include/pa.h compiles as C99 with no CUDA, C++ or framework headers, and a C program
    using every entry point links against the library."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_pa.c"
    calls = "\n".join(f"  (void)&{name};" for name in declared_functions())
    src.write_text(f"""#include "pa.h"
#include <stdio.h>
int main(void) {{
{calls}
  pa_dims d = {{12, 2, 128, 16}};
  printf("%zu %s\\n", pa_decode_workspace_size(&d, 64, 4096, 0), pa_status_string(PA_ERR_RANGE));
  return 0;
}}
""")
    exe = tmp_path / "use_pa"
    lib = Path(L._name)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-pedantic", f"-I{ROOT / 'include'}",
                        str(src), str(lib), f"-Wl,-rpath,{lib.parent}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    size, status = out.stdout.split(maxsplit=1)
    assert int(size) > 0 and status.startswith("PA_ERR_RANGE")


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in include/ but not exported"


def dims(hq=12, hkv=2, d=128, b=16):
    from paged_kv_cache_244_gb300 import binding
    return binding.make_dims(hq, hkv, d, b)


P = ctypes.c_void_p
OK_PTR = P(0x10000)        # 16-byte aligned stand-in pointers: never dereferenced on error paths
MIS_PTR = P(0x10008)


def decode_call(L, d=None, S=2, q=OK_PTR, kc=OK_PTR, vc=OK_PTR, nb=16, bt=OK_PTR, maxb=4,
                ctx=OK_PTR, maxctx=40, scale=0.088, part=0, ws=OK_PTR, wsb=1 << 30, out=OK_PTR):
    d = dims() if d is None else d
    return L.pa_decode(ctypes.byref(d) if d is not False else None, S, q, kc, vc, nb, bt, maxb,
                       ctx, maxctx, scale, part, ws, wsb, out, None)


def test_decode_rejects_bad_arguments_on_the_host(L):
    from paged_kv_cache_244_gb300 import binding as b
    assert decode_call(L, d=False) == b.PA_ERR_NULL
    assert decode_call(L, d=dims(d=64)) == b.PA_ERR_SHAPE
    assert decode_call(L, d=dims(b=32)) == b.PA_ERR_SHAPE
    assert decode_call(L, d=dims(hq=12, hkv=5)) == b.PA_ERR_SHAPE
    assert decode_call(L, d=dims(hq=18, hkv=2)) == b.PA_ERR_SHAPE      # group of 9 > 8
    assert decode_call(L, d=dims(hq=8194, hkv=4097)) == b.PA_ERR_SHAPE  # more KV heads than 4096
    assert decode_call(L, S=-1) == b.PA_ERR_RANGE
    assert decode_call(L, S=0) == b.PA_OK                              # no-op
    for kw in ("q", "kc", "vc", "bt", "ctx", "out"):
        assert decode_call(L, **{kw: None}) == b.PA_ERR_NULL, kw
    assert decode_call(L, maxctx=0) == b.PA_ERR_RANGE
    assert decode_call(L, maxctx=65, maxb=4) == b.PA_ERR_RANGE         # > max_blocks * 16
    assert decode_call(L, part=24) == b.PA_ERR_RANGE                   # not a multiple of 16
    assert decode_call(L, scale=0.0) == b.PA_ERR_RANGE
    assert decode_call(L, scale=float("nan")) == b.PA_ERR_RANGE
    assert decode_call(L, maxctx=40, maxb=4, part=16, wsb=100) == b.PA_ERR_WORKSPACE
    assert decode_call(L, maxctx=40, maxb=4, part=16, ws=None) == b.PA_ERR_WORKSPACE
    assert decode_call(L, maxctx=40, maxb=4, part=64, ws=None) == b.PA_ERR_WORKSPACE
    assert decode_call(L, maxctx=40, maxb=4, part=64, wsb=(3 + 4) * 6 * 520 - 1) == b.PA_ERR_WORKSPACE
    assert decode_call(L, S=8193) == b.PA_ERR_RANGE
    for kw in ("q", "kc", "vc", "bt", "ctx", "out", "ws"):
        assert decode_call(L, **{kw: MIS_PTR}) == b.PA_ERR_ALIGN, kw


def test_decode_step_rejects_bad_arguments_on_the_host(L):
    from paged_kv_cache_244_gb300 import binding as b

    def call(d=None, S=2, maxpos=64, nb=16, maxb=4, maxctx=40, scale=0.088, part=0, wsb=1 << 30,
             flags=0, **ptrs):
        a = dict(q=OK_PTR, k=OK_PTR, v=OK_PTR, cs=OK_PTR, kc=OK_PTR, vc=OK_PTR, bt=OK_PTR,
                 ctx=OK_PTR, ws=OK_PTR, out=OK_PTR)
        a.update(ptrs)
        d = dims() if d is None else d
        return L.pa_decode_step(ctypes.byref(d), S, a["q"], a["k"], a["v"], a["cs"], maxpos,
                                a["kc"], a["vc"], nb, a["bt"], maxb, a["ctx"], maxctx, scale, part,
                                a["ws"], wsb, a["out"], flags, None)

    assert call(flags=2) == b.PA_ERR_RANGE                              # unknown flag bit
    assert call(flags=b.PA_STEP_EARLY_METADATA | 0x100) == b.PA_ERR_RANGE

    assert call(d=dims(d=64)) == b.PA_ERR_SHAPE
    assert call(S=-1) == b.PA_ERR_RANGE
    assert call(S=0) == b.PA_OK
    assert call(S=8193) == b.PA_ERR_RANGE
    for kw in ("q", "k", "v", "cs", "kc", "vc", "bt", "ctx", "out"):
        assert call(**{kw: None}) == b.PA_ERR_NULL, kw
    for kw in ("q", "k", "v", "cs", "kc", "vc", "bt", "ctx", "out", "ws"):
        assert call(**{kw: MIS_PTR}) == b.PA_ERR_ALIGN, kw
    assert call(maxpos=0) == b.PA_ERR_RANGE
    assert call(maxctx=65) == b.PA_ERR_RANGE
    assert call(part=24) == b.PA_ERR_RANGE
    assert call(scale=-1.0) == b.PA_ERR_RANGE
    assert call(part=16, wsb=100) == b.PA_ERR_WORKSPACE


def test_copy_blocks_rejects_bad_arguments_on_the_host(L):
    from paged_kv_cache_244_gb300 import binding as b
    arr = ctypes.c_void_p * 4

    def call(d=None, n=2, nsrc=8, ndst=8, npairs=3, src=None, dst=None, pairs=OK_PTR):
        src = arr(OK_PTR, OK_PTR, OK_PTR, OK_PTR) if src is None else src
        dst = arr(OK_PTR, OK_PTR, OK_PTR, OK_PTR) if dst is None else dst
        d = dims(2, 2) if d is None else d
        return L.pa_copy_blocks(ctypes.byref(d), n, ctypes.cast(src, ctypes.c_void_p), nsrc,
                                ctypes.cast(dst, ctypes.c_void_p), ndst, pairs, npairs, None)

    assert call(d=dims(2, 2, d=64)) == b.PA_ERR_SHAPE
    assert call(npairs=-1) == b.PA_ERR_RANGE
    assert call(npairs=0) == b.PA_OK
    assert call(n=0) == b.PA_ERR_RANGE
    assert call(n=b.PA_MAX_BLOCK_CACHES + 1) == b.PA_ERR_RANGE
    assert call(nsrc=0) == b.PA_ERR_RANGE
    assert call(ndst=0) == b.PA_ERR_RANGE
    assert call(pairs=None) == b.PA_ERR_NULL
    assert call(src=arr(OK_PTR, None, OK_PTR, OK_PTR)) == b.PA_ERR_NULL
    assert call(dst=arr(OK_PTR, MIS_PTR, OK_PTR, OK_PTR)) == b.PA_ERR_ALIGN
    assert call(pairs=P(0x10004)) == b.PA_ERR_ALIGN
    assert L.pa_copy_blocks(ctypes.byref(dims(2, 2)), 2, None, 8, None, 8, OK_PTR, 1, None) == b.PA_ERR_NULL


def test_fp8_entry_points_reject_bad_arguments_on_the_host(L):
    from paged_kv_cache_244_gb300 import binding as b
    d = dims()

    def dec(ks=OK_PTR, vs=OK_PTR, S=2, **kw):
        a = dict(q=OK_PTR, kc=OK_PTR, vc=OK_PTR, bt=OK_PTR, ctx=OK_PTR, ws=OK_PTR, out=OK_PTR)
        a.update(kw)
        return L.pa_decode_fp8(ctypes.byref(d), S, a["q"], a["kc"], a["vc"], ks, vs, 16, a["bt"], 4,
                               a["ctx"], 40, 0.088, 0, a["ws"], 1 << 30, a["out"], None)

    assert dec(S=0) == b.PA_OK
    assert dec(ks=None) == b.PA_ERR_NULL and dec(vs=None) == b.PA_ERR_NULL
    assert dec(ks=MIS_PTR) == b.PA_ERR_ALIGN
    assert dec(q=None) == b.PA_ERR_NULL and dec(kc=MIS_PTR) == b.PA_ERR_ALIGN
    assert dec(S=-1) == b.PA_ERR_RANGE

    def store(ks=OK_PTR, vs=OK_PTR, T=3):
        return L.pa_rope_kv_store_fp8(ctypes.byref(d), T, OK_PTR, OK_PTR, OK_PTR, OK_PTR, OK_PTR, 64,
                                      OK_PTR, OK_PTR, OK_PTR, 16, ks, vs, None)

    assert store(T=0) == b.PA_OK
    assert store(ks=None) == b.PA_ERR_NULL and store(vs=MIS_PTR) == b.PA_ERR_ALIGN

    def step(ks=OK_PTR, vs=OK_PTR, S=2, k=OK_PTR, flags=0):
        return L.pa_decode_step_fp8(ctypes.byref(d), S, OK_PTR, k, OK_PTR, OK_PTR, 64, OK_PTR, OK_PTR,
                                    ks, vs, 16, OK_PTR, 4, OK_PTR, 40, 0.088, 0, OK_PTR, 1 << 30,
                                    OK_PTR, flags, None)

    assert step(flags=4) == b.PA_ERR_RANGE

    assert step(S=0) == b.PA_OK
    assert step(ks=None) == b.PA_ERR_NULL and step(vs=MIS_PTR) == b.PA_ERR_ALIGN
    assert step(k=None) == b.PA_ERR_NULL


def test_prefill_rejects_bad_arguments_on_the_host(L):
    from paged_kv_cache_244_gb300 import binding as b

    def call(d=None, S=2, T=40, maxq=32, maxctx=64, maxb=4, scale=0.088, **ptrs):
        a = dict(q=OK_PTR, qs=OK_PTR, kc=OK_PTR, vc=OK_PTR, bt=OK_PTR, ctx=OK_PTR, out=OK_PTR)
        a.update(ptrs)
        d = dims() if d is None else d
        return L.pa_prefill(ctypes.byref(d), S, T, a["q"], a["qs"], maxq, a["kc"], a["vc"], 16,
                            a["bt"], maxb, a["ctx"], maxctx, scale, a["out"], None)

    assert call(d=dims(d=64)) == b.PA_ERR_SHAPE
    assert call(S=-1) == b.PA_ERR_RANGE and call(T=-1) == b.PA_ERR_RANGE
    assert call(S=0) == b.PA_OK and call(T=0) == b.PA_OK
    for kw in ("q", "qs", "kc", "vc", "bt", "ctx", "out"):
        assert call(**{kw: None}) == b.PA_ERR_NULL, kw
        assert call(**{kw: MIS_PTR}) == b.PA_ERR_ALIGN, kw
    assert call(maxq=0) == b.PA_ERR_RANGE
    assert call(maxq=65) == b.PA_ERR_RANGE                  # above max_context_len
    assert call(maxctx=65) == b.PA_ERR_RANGE                # above max_blocks * 16
    assert call(S=40000) == b.PA_ERR_RANGE                  # S * Hkv > 65535
    assert call(scale=0.0) == b.PA_ERR_RANGE


def test_rope_kv_store_rejects_bad_arguments_on_the_host(L):
    from paged_kv_cache_244_gb300 import binding as b

    def call(d=None, T=3, maxpos=64, nb=16, **ptrs):
        args = dict(q=OK_PTR, k=OK_PTR, v=OK_PTR, pos=OK_PTR, cs=OK_PTR, slot=OK_PTR,
                    kc=OK_PTR, vc=OK_PTR)
        args.update(ptrs)
        d = dims() if d is None else d
        return L.pa_rope_kv_store(ctypes.byref(d), T, args["q"], args["k"], args["v"], args["pos"],
                                  args["cs"], maxpos, args["slot"], args["kc"], args["vc"], nb, None)

    assert call(d=dims(d=96)) == b.PA_ERR_SHAPE
    assert call(T=-1) == b.PA_ERR_RANGE
    assert call(T=0) == b.PA_OK
    for kw in ("q", "k", "v", "pos", "cs", "slot", "kc", "vc"):
        assert call(**{kw: None}) == b.PA_ERR_NULL, kw
        assert call(**{kw: MIS_PTR}) == b.PA_ERR_ALIGN, kw
    assert call(maxpos=0) == b.PA_ERR_RANGE
    assert call(nb=0) == b.PA_ERR_RANGE


def test_partition_choice_and_workspace_size(L):
    from paged_kv_cache_244_gb300 import binding as b
    # the request is validated and echoed: 0 = even split, else a multiple of 16 tokens
    assert b.decode_partition_tokens(12, 2, 2, 40) == 0
    assert b.decode_partition_tokens(12, 2, 4, 32768, 512) == 512
    for bad in (100, -16):
        with pytest.raises(b.PaError):
            b.decode_partition_tokens(12, 2, 4, 32768, bad)
    with pytest.raises(b.PaError):
        b.decode_partition_tokens(12, 2, 8193, 64)              # more sequences than supported
    # workspace: (ranges + segments * partitions) * G rows of (D + 2) floats, ranges <=
    # min(2048, ceil(jobs / 2))
    row = 130 * 4
    # 4 x 32768 tokens, 512-token partitions: 2048 ranges + 8 segments x 64 partitions
    assert b.decode_workspace_size(12, 2, 4, 32768, 512) == (2048 + 8 * 64) * 6 * row
    # 2 x 40 tokens: 12 jobs -> 6 ranges; 64-token partitions: one per segment
    assert b.decode_workspace_size(12, 2, 2, 40, 64) == (6 + 4) * 6 * row
    assert b.decode_workspace_size(12, 2, 2, 40) == (6 + 4) * 6 * row
    # 16-token partitions: 3 per segment
    assert b.decode_workspace_size(12, 2, 2, 40, 16) == (6 + 4 * 3) * 6 * row
    assert b.decode_workspace_size(12, 2, 64, 4096) == (2048 + 128) * 6 * row
    assert b.decode_workspace_size(12, 2, 4, 32768, 100) == 0


def test_selftest_rejects_bad_limits_on_the_host(L):
    from paged_kv_cache_244_gb300 import binding as b
    assert L.pa_selftest_wait_timeout(0, None) == b.PA_ERR_RANGE
    assert L.pa_selftest_wait_timeout(2000000, None) == b.PA_ERR_RANGE


def test_stage_copy_checks_its_arguments_on_the_host(L):
    """Null, alignment and size checks come before any CUDA call (none is made here)."""
    import ctypes
    from paged_kv_cache_244_gb300 import binding as b
    buf = (ctypes.c_ubyte * 96)()
    base = ctypes.addressof(buf)
    a16 = base + (-base) % 16                         # a 16-byte aligned address inside buf
    vp = ctypes.c_void_p
    assert L.pa_stage_copy(vp(a16), vp(a16 + 32), 0, None) == b.PA_OK            # no-op
    assert L.pa_stage_copy(None, vp(a16), 16, None) == b.PA_ERR_NULL
    assert L.pa_stage_copy(vp(a16), None, 16, None) == b.PA_ERR_NULL
    assert L.pa_stage_copy(vp(a16 + 8), vp(a16 + 32), 16, None) == b.PA_ERR_ALIGN
    assert L.pa_stage_copy(vp(a16), vp(a16 + 40), 16, None) == b.PA_ERR_ALIGN
    assert L.pa_stage_copy(vp(a16), vp(a16 + 32), 24, None) == b.PA_ERR_ALIGN


def test_timing_jitter_range_is_checked_on_the_host(L):
    from paged_kv_cache_244_gb300 import binding as b
    assert L.pa_set_timing_jitter(1000001, 0) == b.PA_ERR_RANGE


def test_status_strings(L):
    from paged_kv_cache_244_gb300 import binding as b
    for code in range(0, -9, -1):
        assert b.status_string(code).startswith("PA_")
    assert b.status_string(7) == "unknown pa status"
