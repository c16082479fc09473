"""The C ABI from plain C: tests/abi_from_c.c is compiled with gcc as C11
against include/hb.h and libhb.so and run on the host (no GPU); its trace of
status names, a host-only plan, argument errors and a batch-builder run must
equal the same calls made through the Python binding."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from _hbutil import ROOT, host_batch, lib


def _python_trace(hb):
    L = hb.load()
    out = [f"status {s} {L.hb_status_string(s).decode()}" for s in range(9)]
    b, ql, cl = host_batch(hb, [(1, 40), (5, 9), (40, 100)], hq=32, hkv=8, d=128,
                           max_pages=7, num_pages=12)
    pb, wb = hb.hb_plan_sizes(b, ql, cl, 152)
    out.append(f"sizes {pb} {wb}")
    plan, _ = hb.hb_plan(b, ql, cl, 152, upload=False)
    out.append("plan " + bytes(plan[:pb]).hex())
    for name, args in (("bad_row", (b, np.array([1, 10, 40], np.int32), cl)),
                       ("null_batch", (None, ql, cl))):
        if args[0] is None:
            st = L.hb_plan(None, hb._ptr(ql), hb._ptr(cl), 152, None,
                           hb.ctypes.byref(hb.ctypes.c_size_t(0)), None,
                           hb.ctypes.byref(hb.ctypes.c_size_t(0)), None)
        else:
            with pytest.raises(hb.HbError) as e:
                hb.hb_plan_sizes(*args, 152)
            st = e.value.status
        out.append(f"{name} {hb.STATUS_NAMES[st]} {int(bool(L.hb_last_error()))}")
    bld = hb.Builder(24, 16, 10, 4)
    for rid, p, m in ((7, 30, 2), (3, 5, 1), (9, 12, 3)):
        bld.add_request(rid, p, m)
    with pytest.raises(hb.HbError) as e:
        bld.add_request(7, 4, 1)
    out.append(f"duplicate {hb.STATUS_NAMES[e.value.status]}")
    for it in range(16):
        st = bld.step()
        if st is None:
            break
        out.append(f"step {it} rows {len(st['q_len'])} over {int(st['over_budget'])}")
        for r in range(len(st["q_len"])):
            pages = " ".join(str(int(x)) for x in st["block_table"][r])
            out.append(f"  row {int(st['ids'][r])} kind {int(st['kind'][r])} q "
                       f"{int(st['q_len'][r])} ctx {int(st['context_len'][r])} pages {pages}")
        fin = bld.complete()
        out.append("  finished" + "".join(f" {x}" for x in fin))
    w, r, f = bld.counts()
    out.append(f"counts {w} {r} {f}")
    bld.close()
    return out


def test_header_compiles_as_c_and_matches_the_binding(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    hb = lib()
    so = hb.lib_path()
    exe = str(tmp_path / "abi_from_c")
    cmd = [gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-O1",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "abi_from_c.c"),
           so, "-Wl,-rpath," + os.path.dirname(so), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    got = r.stdout.splitlines()
    want = _python_trace(hb)
    assert got == want
    # the trace covers what it claims to
    assert any(ln.startswith("plan ") and len(ln) > 400 for ln in got)
    assert sum(ln.startswith("step ") for ln in got) >= 3
    assert got[-1] == "counts 0 0 10"
