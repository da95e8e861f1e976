"""The C ABI library: builds for sm_103a, loads, exports every declared entry point, and
rejects bad arguments on the host before touching CUDA.  No GPU needed."""

import ctypes
import os
import re
import subprocess

import pytest

from speculative_decoding_draft_kv_gb300 import build as B
from speculative_decoding_draft_kv_gb300 import ring as R

HEADER = os.path.join(B.INCLUDE, "dflash_ring.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return R.library()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(ring_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_binding_names():
    assert _declared() == sorted(R.EXPORTED)


def test_shared_object_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in _declared():
        assert name in syms, name
        assert getattr(lib, name) is not None


def test_build_targets_sm_103a_only():
    assert B.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def _init_rc(**kw):
    p = dict(cap=64, q_len=8, head_dim=128, n_head_kv=8, n_head=32, n_layer=1,
             rope_theta=1e6, n_seq=1, swa_window=0, bulk_chunk=0, tiles_per_split=0,
             max_cluster=0)
    p.update(kw)
    h = ctypes.c_void_p()
    rc = R.library().ring_init_ex(ctypes.byref(h), ctypes.byref(R.RingParams(**p)))
    return rc, h


@pytest.mark.parametrize("bad", [
    dict(cap=0), dict(q_len=-1), dict(head_dim=64), dict(n_head=30), dict(n_layer=0),
    dict(rope_theta=0.0), dict(n_head=64),            # 8 heads per kv head * 8 queries > 32 rows
    dict(swa_window=-3), dict(cap=2**30),
])
def test_init_rejects_bad_shapes_on_the_host(lib, bad):
    rc, h = _init_rc(**bad)
    assert rc == R.RING_EINVAL and not h.value
    assert R.ring_last_error(None)


def test_null_handles_are_rejected(lib):
    assert lib.ring_destroy(None) == R.RING_OK
    assert lib.ring_get_geometry(None, None) == R.RING_EINVAL
    assert lib.ring_begin_step(None, None, None, None, None, None, 0, None) == R.RING_EINVAL
    assert lib.ring_attend(None, 0, 0, None, None, None, None, None) == R.RING_EINVAL
    assert lib.ring_launch_count(None) == 0
    assert lib.ring_init_ex(None, None) == R.RING_EINVAL
    assert isinstance(R.ring_last_error(None), str)


def test_product_path_never_imports_the_oracle():
    pkg = os.path.dirname(B.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cuh")):
                src = open(os.path.join(root, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f


def test_header_is_plain_c_and_struct_layouts_match_the_binding(tmp_path):
    """The header compiles as C99 (no C++ or CUDA types in the signatures), and every
    struct has the size and field offsets the ctypes binding assumes."""
    import shutil
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"ring_params": R.RingParams, "ring_geometry": R.RingGeometry,
               "ring_profile": R.RingProfile, "ring_producer": R.RingProducer,
               "ring_attend_static_args": R.RingAttendStaticArgs}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "dflash_ring.h"',
             'int main(void) {']
    for cname, py in structs.items():
        lines.append(f'    printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'    printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ['    return 0;', '}']
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", B.INCLUDE, str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {tuple(line.split()[:2]): int(line.split()[2]) for line in out if line.strip()}
    for cname, py in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for fname, _ in py._fields_:
            assert got[(cname, fname)] == getattr(py, fname).offset, (cname, fname)
