"""Host check (no GPU): the Python binding's ctypes structures have the same
size and field offsets as the C declarations in include/attn_bwd.h (a small C
program built here with the host compiler prints them)."""

import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _c_layout(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    exe = tmp_path / "abi_layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
                    os.path.join(ROOT, "tests", "native", "abi_layout.c"), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    return {k: int(v) for k, v in (line.split() for line in out.splitlines())}


def test_ctypes_structs_match_the_header(tmp_path):
    import __graft_entry__
    __graft_entry__.build()
    import attention_backward_attn_gb300 as ab
    c = _c_layout(tmp_path)
    for cname, py in (("attn_problem_t", ab.Problem), ("attn_mask_t", ab.Mask),
                      ("attn_sparse_t", ab.Sparse)):
        assert ctypes.sizeof(py) == c[cname], cname
        for name, _ in py._fields_:
            assert getattr(py, name).offset == c[f"{cname}.{name}"], (cname, name)
