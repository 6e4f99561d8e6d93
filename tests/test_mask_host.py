"""Host checks (no GPU): the library's mask arithmetic, element by element,
against the oracle's mask ("22_sink_tokens_fmha.py" mask builders, with the
library's (window_left, window_right, num_sink, bottom_right) reading).

* The C ABI's tile classes with 1 x 1 tiles are the element mask as the
  kernels' host side sees it (descriptor conversion, tile_any / tile_full).
* The predicates of csrc/mask.h (mask_live, and the row / column ranges the
  CUDA-core kernels walk) are dumped by a small host program
  (tests/native/mask_elements.cpp).

Shapes: every dense benchmark workload, ragged and misaligned ones, and 300
random draws. The device side of the same decisions is checked in
tests/test_gpu_masks.py.
"""

import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (Sq, Sk, window_left, window_right, num_sink, bottom_right)
WORKLOAD_MASKS = [
    (64, 64, -1, -1, 0, 0),
    (1024, 1024, -1, 0, 0, 0),
    (2048, 2048, -1, -1, 0, 0),
    (8192, 8192, 1023, 0, 4, 0),
]
RAGGED_MASKS = [
    (1000, 1000, -1, 0, 0, 0), (1, 1, -1, 0, 0, 0), (200, 330, -1, 0, 0, 1),
    (330, 200, -1, 0, 0, 1), (330, 200, 50, 7, 0, 1), (129, 127, 30, 0, 5, 0),
    (300, 5, -1, 0, 2, 0), (5, 300, -1, -1, 200, 0), (640, 640, 0, 0, 0, 0),
    (384, 512, 127, 128, 1, 0), (256, 256, 10, 0, 130, 0), (700, 450, 1023, 0, 4, 1),
]


def _random_masks(n=300, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        Sq, Sk = int(rng.integers(1, 400)), int(rng.integers(1, 400))
        wl = int(rng.choice([-1, int(rng.integers(0, 300))]))
        wr = int(rng.choice([-1, 0, int(rng.integers(0, 150))]))
        ns = int(rng.choice([0, 0, int(rng.integers(1, 100))]))
        out.append((Sq, Sk, wl, wr, ns, int(rng.integers(0, 2))))
    return out


def _ref(case):
    Sq, Sk, wl, wr, ns, br = case
    return oracle.live_mask(Sq, Sk, wl, wr, ns, bool(br))


@pytest.fixture(scope="module")
def ab():
    import __graft_entry__
    __graft_entry__.build()
    import attention_backward_attn_gb300 as mod
    return mod


@pytest.mark.parametrize("group", ["workloads", "ragged", "random"])
def test_abi_element_classes_equal_oracle_mask(ab, group):
    cases = {"workloads": WORKLOAD_MASKS, "ragged": RAGGED_MASKS,
             "random": _random_masks()}[group]
    for case in cases:
        Sq, Sk, wl, wr, ns, br = case
        buf = np.full(Sq * Sk, -1, dtype=np.int8)
        code = ab.lib.attn_mask_tile_classes(ctypes.byref(ab.Mask(wl, wr, ns, br)), Sq, Sk, 1, 1,
                                             buf.ctypes.data)
        assert code == 0
        got = buf.reshape(Sq, Sk)
        assert not (got == 1).any(), case  # a 1 x 1 tile is all live or all dead
        assert np.array_equal(got == 2, _ref(case)), case


@pytest.fixture(scope="module")
def dumper(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path_factory.mktemp("mask") / "mask_elements"
    src = os.path.join(ROOT, "tests", "native", "mask_elements.cpp")
    inc = os.path.join(ROOT, "attention_backward_attn_gb300", "csrc")
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", inc, src, "-o", str(exe)], check=True)
    return str(exe)


@pytest.mark.parametrize("group", ["workloads", "ragged", "random"])
def test_mask_predicates_equal_oracle_mask(dumper, group):
    cases = {"workloads": WORKLOAD_MASKS, "ragged": RAGGED_MASKS,
             "random": _random_masks()}[group]
    text = "".join(" ".join(map(str, c)) + "\n" for c in cases)
    out = subprocess.run([dumper], input=text.encode(), capture_output=True, check=True).stdout
    off = 0
    for case in cases:
        Sq, Sk = case[0], case[1]
        ref = _ref(case)
        for plane in ("mask_live", "row ranges", "column ranges"):
            got = np.frombuffer(out, dtype=np.uint8, count=Sq * Sk, offset=off).reshape(Sq, Sk)
            off += Sq * Sk
            assert np.array_equal(got.astype(bool), ref), (plane, case)
    assert off == len(out)
