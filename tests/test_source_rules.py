"""Source-level rules of the device code that keep a failing run from hanging or
faulting the GPU, checked by reading csrc/ (CPU only):

* no trap, breakpoint or device-side assert: failures travel through the
  status word;
* the raw mbarrier try_wait is issued by one helper, and the only loops around
  it are the two bounded waits (a time limit on %globaltimer);
* the only other endless-looking loops are the bounded waits themselves and the
  replay draw's 128-way search, whose interval shrinks every round;
* every kernel that allocates tensor memory releases it after a CTA-wide
  barrier, on every path (the dealloc follows the kernel's last __syncthreads).
"""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "rl_experience_collection_gb300", "csrc")


def _sources():
    out = {}
    for p in sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))):
        src = open(p).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        out[os.path.basename(p)] = src
    return out


def _body(src, signature_regex):
    """The brace-balanced body of the first function whose header matches."""
    m = re.search(signature_regex, src)
    assert m, signature_regex
    i = src.index("{", m.end())
    depth = 0
    for j in range(i, len(src)):
        depth += {"{": 1, "}": -1}.get(src[j], 0)
        if depth == 0:
            return src[i:j + 1]
    raise AssertionError("unbalanced braces")


def test_no_trap_breakpoint_or_device_assert():
    for name, src in _sources().items():
        assert "__trap" not in src and not re.search(r"\btrap\s*;", src), name
        assert "brkpt" not in src, name
        assert not re.search(r"(?<!static_)\bassert\s*\(", src), name


def test_raw_try_wait_only_inside_bounded_waits():
    srcs = _sources()
    for name, src in srcs.items():
        if re.search(r"mbarrier\.(try_wait|test_wait)", src):
            assert name == "umma.cuh", name
    bounded = {("umma.cuh", r"bool\s+mbar_wait\s*\("), ("dqn.cu", r"void\s+mbar_wait_drain\s*\(")}
    allowed = 0
    for name, sig in bounded:
        body = _body(srcs[name], sig)
        assert "global_ns()" in body and re.search(r"global_ns\(\)\s*-\s*t0\s*>", body), name
        allowed += body.count("mbar_try_wait(")
    calls = sum(src.count("mbar_try_wait(") for src in srcs.values())
    definitions = len(re.findall(r"bool\s+mbar_try_wait\s*\(", srcs["umma.cuh"]))
    assert calls - definitions == allowed


def test_endless_loop_forms_are_the_known_bounded_ones():
    found = {}
    for name, src in _sources().items():
        n = len(re.findall(r"while\s*\(\s*(true|1)\s*\)|for\s*\(\s*;\s*;\s*\)", src))
        if n:
            found[name] = n
    # umma.cuh: mbar_wait (time limit); per.cu: the draw's search (interval shrinks)
    assert found == {"umma.cuh": 1, "per.cu": 1}, found
    assert re.search(r"while\s*\(\s*true\s*\)", _body(_sources()["umma.cuh"], r"bool\s+mbar_wait\s*\("))
    search = _body(_sources()["per.cu"], r"void\s+__launch_bounds__\(kSampleWarps \* 32\) sample_kernel\s*\(")
    assert "if (span <= 1) break;" in search


def test_tensor_memory_released_after_the_last_cta_barrier():
    for name, src in _sources().items():
        if name == "umma.cuh":
            continue
        allocs = src.count("tmem_alloc(")
        assert allocs == src.count("tmem_dealloc("), name
        for m in re.finditer(r"tmem_dealloc\(", src):
            before = src[:m.start()]
            last_sync = before.rfind("__syncthreads();")
            assert last_sync >= 0, name
            # nothing between that barrier and the dealloc waits or returns
            gap = before[last_sync:]
            assert "return" not in gap and "mbar_wait" not in gap and "while" not in gap, name
