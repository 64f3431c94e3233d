"""How bench.py ties its roofline `traffic` figures to the committed ncu
summaries: a summary counts only while the kernel's code (comments and
whitespace aside) is the code it was captured from."""
import glob
import importlib.util
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


CODE = """// kernel header
__global__ void k(float *x, int n) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;   /* one element per thread */
  if (i < n) x[i] *= 2.0f;
}
"""


def test_code_hash_ignores_comments_and_whitespace(bench, tmp_path):
    a, b, c = tmp_path / "a.cu", tmp_path / "b.cu", tmp_path / "c.cu"
    a.write_text(CODE)
    # the same code with other comments and another layout
    b.write_text("/* new\n   block comment */\n__global__ void k(float *x,\n   int n) {\n"
                 "  int i = blockIdx.x * blockDim.x + threadIdx.x; // index\n"
                 "  if (i < n)   x[i] *= 2.0f;   // scale\n}\n")
    c.write_text(CODE.replace("2.0f", "3.0f"))
    assert bench.code_hash(str(a)) == bench.code_hash(str(b))
    assert bench.code_hash(str(a)) != bench.code_hash(str(c))


def _summaries():
    out = []
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        text = open(path).read()
        h = re.search(r"^code_sha256_prefix: ([0-9a-f]+)$", text, re.M)
        if h:
            out.append((path, text, h.group(1)))
    return out


def test_every_kernel_summary_names_its_figures_and_command():
    found = _summaries()
    assert found, "no kernel summaries under profiles/"
    for path, text, prefix in found:
        name = os.path.basename(path)
        assert len(prefix) >= 12, name
        assert re.search(r"^traffic_bytes_per_launch: \d+$", text, re.M), name
        cmd = [ln for ln in text.splitlines() if ln.startswith("    ") and " ncu " in ln]   # the command block
        assert cmd and all("--clock-control none" in ln for ln in cmd), name
        assert re.search(r"sparse_kv_offload_gb300/csrc/\w+\.cu", text), name


def test_traffic_counts_only_for_the_captured_code(bench, monkeypatch):
    by_kernel = {kernel: stage for stage, (kernel, _src) in bench.KERNEL_SOURCE.items()}
    checked = 0
    for path, text, prefix in _summaries():
        name = os.path.basename(path)[:-3]
        kernel = max((k for k in by_kernel if name.startswith(k + "_")), key=len, default=None)
        if kernel is None:
            continue
        workload = name[len(kernel) + 1:]
        want = int(re.search(r"^traffic_bytes_per_launch: (\d+)$", text, re.M).group(1))
        monkeypatch.setattr(bench, "code_hash", lambda *p, pre=prefix: pre + "0" * 8)
        assert bench.profiled_traffic(by_kernel[kernel], workload) == want, name
        monkeypatch.setattr(bench, "code_hash", lambda *p, pre=prefix: ("f" if pre[0] != "f" else "0") + pre[1:])
        assert bench.profiled_traffic(by_kernel[kernel], workload) is None, name
        checked += 1
    assert checked >= 1
