"""Register and local-memory budget of every kernel, from the assembler's own report
(``-Xptxas -v``), checked at build time on the CPU.

* No kernel spills registers to local memory.
* Every instantiation of the tcgen05 kernel compiles to exactly its launch
  register count (168 per thread at 384 threads). Its control warpgroup drops to
  88 registers and its two softmax warpgroups rise to 208 with setmaxnreg, and
  88 * 128 + 208 * 256 = 64 512 = 168 * 384: the split draws exactly the
  registers the launch holds. The launcher refuses any other count at run time;
  this catches it at build time, reading the counts from the kernel source.
"""
import os
import re
import shutil
import subprocess

import pytest

from vision_encoder_varlen_gb300 import _build

_ENTRY = re.compile(r"Compiling entry function '([^']+)'.*?(\d+) bytes stack frame, (\d+) bytes spill stores, "
                    r"(\d+) bytes spill loads\s*\nptxas info\s*: Used (\d+) registers", re.S)


def _demangle(names):
    tool = shutil.which("c++filt")
    if not tool:
        return list(names)
    r = subprocess.run([tool], input="\n".join(names), capture_output=True, text=True)
    return r.stdout.splitlines() if r.returncode == 0 else list(names)


@pytest.fixture(scope="module")
def kernels(tmp_path_factory):
    try:
        results = _build.compile_all(str(tmp_path_factory.mktemp("ptxas")), ptxas_info=True)
    except RuntimeError as e:
        if "nvcc not found" in str(e):
            pytest.skip(str(e))
        raise
    found = []
    for _, log in results:
        for name, stack, spill_st, spill_ld, regs in _ENTRY.findall(log):
            found.append({"mangled": name, "regs": int(regs), "stack": int(stack),
                          "spill_stores": int(spill_st), "spill_loads": int(spill_ld)})
    for k, dem in zip(found, _demangle([k["mangled"] for k in found])):
        k["name"] = dem
    return found


def test_every_kernel_is_reported(kernels):
    names = " ".join(k["name"] for k in kernels)
    for kern in ("attn_long_kernel", "attn_tiny_kernel", "qk_norm_rope_kernel",
                 "qk_norm_rope_staged_kernel", "rope_freqs_kernel", "rope_table_kernel", "schedule_kernel"):
        assert kern in names, kern


def test_no_kernel_spills(kernels):
    spilled = [(k["name"], k["spill_stores"], k["spill_loads"]) for k in kernels
               if k["spill_stores"] or k["spill_loads"]]
    assert not spilled, spilled


def _constant(src: str, name: str) -> int:
    m = re.search(rf"constexpr int {name} = (\d+);", src)
    assert m, name
    return int(m.group(1))


def test_tcgen05_kernel_register_count_matches_its_split(kernels):
    with open(os.path.join(_build.CSRC, "attn_long.cu")) as f:
        src = f.read()
    threads, launch = _constant(src, "kThreads"), _constant(src, "kLaunchRegs")
    # one control warpgroup and the rest softmax warpgroups, 128 threads each: neither split (the
    # plain one, and the one of the variant that rotates raw Q) may draw more than the launch
    # holds (setmaxnreg.inc would wait for registers forever)
    for ctrl_name, softmax_name in (("kCtrlRegs", "kSoftmaxRegs"), ("kCtrlRegsFQ", "kSoftmaxRegsFQ")):
        ctrl, softmax = _constant(src, ctrl_name), _constant(src, softmax_name)
        assert ctrl * 128 + softmax * (threads - 128) <= launch * threads
        assert ctrl % 8 == 0 and softmax % 8 == 0
    assert launch * threads <= 65536 and launch % 8 == 0
    long_k = [k for k in kernels if "attn_long_kernel" in k["name"]]
    assert long_k
    assert all(k["regs"] == launch for k in long_k), [(k["name"], k["regs"]) for k in long_k]
