"""The decode kernel's pair plans, checked on the host: for every width and
group, the entries of a thread's chunk name every code exactly once, and
(affine widths) each code sits where its fp16 half expects it -- code lo at
bit plo and code hi at bit 16 + phi of the 32-bit window that starts at
stream bit S -- with 2^p * q < 1024, so that (window & mask) | 1024 is the
exact fp16 value 1024 + 2^p * q.  A wrong plan entry would mis-assign codes
on the GPU; the GPU parity tests would catch it too, this pins it without a
device."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_SRC = r"""
#include <cstdio>
#include "gemv_impl.cuh"
using namespace qg::gemv;
int main() {
    int bad = 0;
    for (int bits = 2; bits <= 6; bits++) {
        for (int G : {64, 128}) {
            const int nc = G / 4;                 // codes of a thread's chunk
            int seen[64] = {0};
            for (int e = 0; e < nc / 2; e++) {
                const PairE p = plan_entry(bits, nc, e);
                if (p.lo < 0 || p.lo >= nc || p.hi < 0 || p.hi >= nc) { bad++; continue; }
                seen[p.lo]++;
                seen[p.hi]++;
                if (bits == 2) continue;          // codebook: byte-permute lookups, no bit windows
                if (bits * p.lo - p.S != p.plo || bits * p.hi - p.S != 16 + p.phi) {
                    bad++; printf("position b%d g%d e%d\n", bits, G, e);
                }
                if (p.plo < 0 || p.phi < 0 || p.plo + bits > 10 || p.phi + bits > 10) {
                    bad++; printf("exponent b%d g%d e%d\n", bits, G, e);
                }
            }
            for (int c = 0; c < nc; c++)
                if (seen[c] != 1) { bad++; printf("cover b%d g%d c%d x%d\n", bits, G, c, seen[c]); }
        }
    }
    printf(bad ? "FAIL %d\n" : "OK\n", bad);
    return bad ? 1 : 0;
}
"""


def test_pair_plans_cover_every_code_at_its_bit(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    src = tmp_path / "plan_check.cu"
    src.write_text(_SRC)
    exe = tmp_path / "plan_check"
    csrc = os.path.join(ROOT, "bit_weight_only_group_gb300", "csrc")
    r = subprocess.run([nvcc, "-std=c++17", "--expt-relaxed-constexpr", f"-I{ROOT}/include", f"-I{csrc}",
                        "-o", str(exe), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip().endswith("OK"), out.stdout
