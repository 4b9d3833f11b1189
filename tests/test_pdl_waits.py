"""Every kernel that may start early must wait for the kernel before it.

A launch through launch_pdl (or the grouped GEMM's own launch, which sets the same
programmatic-serialization attribute) lets the kernel begin while the previous kernel in the
stream is still running.  Such a kernel must call pdl_wait() before it touches global memory that
an earlier kernel writes or reads.  This test reads the CUDA sources and checks that each kernel
named in a launch_pdl call, and the grouped GEMM, has pdl_wait() in its body.  A kernel launched
early without it would race, silently, with its predecessor.
"""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "moe_expert_ffn_03_gb300", "csrc")


def sources():
    return {os.path.basename(p): open(p).read() for p in sorted(glob.glob(os.path.join(CSRC, "*.cu")))}


def kernel_body(src, name):
    """The body of the __global__ function `name` (template or not), or None."""
    for m in re.finditer(r"__global__[^;{]*?\b" + re.escape(name) + r"\s*\(", src, re.S):
        i = src.index("{", m.end())
        depth, j = 0, i
        while True:
            if src[j] == "{":
                depth += 1
            elif src[j] == "}":
                depth -= 1
                if depth == 0:
                    return src[i:j + 1]
            j += 1
    return None


def early_launched_kernels(srcs):
    names = set()
    for text in srcs.values():
        for m in re.finditer(r"launch_pdl\(\s*([A-Za-z_]\w*)", text):
            names.add(m.group(1))
    return names


def test_every_early_launched_kernel_waits():
    srcs = sources()
    names = early_launched_kernels(srcs)
    assert len(names) >= 10, sorted(names)               # routing, quantizers, combine, dprob
    for name in sorted(names):
        bodies = [b for b in (kernel_body(t, name) for t in srcs.values()) if b is not None]
        assert bodies, f"no __global__ definition of {name}"
        for b in bodies:
            assert "pdl_wait();" in b, f"{name} is launched with launch_pdl but never calls pdl_wait()"


def test_grouped_gemm_waits_before_reading_routing_data():
    src = sources()["gemm.cu"]
    assert "cudaLaunchAttributeProgrammaticStreamSerialization" in src
    body = kernel_body(src, "grouped_gemm_kernel")
    assert body is not None
    wait = body.index("pdl_wait();")
    # the segment table is built from split_sizes, which the routing writes
    assert wait < body.index("args.split_sizes"), "grouped_gemm_kernel reads split_sizes before pdl_wait()"


def test_launch_helper_sets_the_attribute_only_below_the_cta_bound():
    text = open(os.path.join(CSRC, "kernels.cuh")).read()
    assert re.search(r"constexpr int64_t kPdlMaxCtas = \d+;", text)
    assert "cfg.numAttrs = int64_t(grid.x) * grid.y * grid.z <= kPdlMaxCtas ? 1 : 0;" in text
