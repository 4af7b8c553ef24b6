"""CPU tests of the compiled host planners behind the scan's launch: the
segmented scan's plan (segments P of L chunks) and the value-row split.  A small
driver, built with nvcc and linked against the library's own object files,
enumerates plans over batch shapes and SM counts; the checks are the bounds the
kernels rely on: the segment planes fit the workspace's fixed area, pass A fits one
wave of the GPU, and the segments cover every chunk."""
import os
import re
import shutil
import subprocess

import pytest

from kda_prefill_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "kda_prefill_gb300", "csrc")

DRIVER = r"""
#include <cstdio>
#include "kda_internal.h"

int main() {
    static const int sms_list[] = {16, 100, 132, 148, 152, 160};
    float plane = 0.f;
    for (int s : sms_list)
        for (int nl = 1; nl <= 2; ++nl)
            for (int H = 1; H <= 6; ++H)
                for (int mc = 1; mc <= 700; ++mc) {
                    kda::FwdParams p{};
                    p.seg = &plane;
                    p.long_list = nullptr;
                    p.N = nl;
                    p.H = H;
                    p.max_long_chunks = mc;
                    int L = 0;
                    const int P = kda::scan_segments(p, s, &L);
                    std::printf("%d %d %d %d %d %d %d %d\n", s, nl, H, mc, P, L,
                                kda::scan_groups(nl, H, s), kda::scan_groups(nl, H, s, s));
                }
    return 0;
}
"""


@pytest.fixture(scope="module")
def plans(tmp_path_factory):
    nvcc = kbuild.NVCC if shutil.which(kbuild.NVCC) else None
    if nvcc is None:
        pytest.skip("nvcc not available")
    kbuild.build()
    objs = [os.path.join(kbuild.BUILD_DIR, os.path.splitext(s)[0] + ".o") for s in kbuild.SOURCES]
    d = tmp_path_factory.mktemp("plans")
    src, exe = d / "plans.cu", d / "plans"
    src.write_text(DRIVER)
    cmd = [nvcc, "-std=c++17", *kbuild.ARCH, f"-I{os.path.join(ROOT, 'include')}", f"-I{CSRC}",
           str(src), *objs, "-o", str(exe), "-cudart", "static", "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    return [tuple(int(x) for x in line.split()) for line in r.stdout.splitlines()]


def _seg_planes():
    src = open(os.path.join(CSRC, "kda_internal.h")).read()
    return int(re.search(r"constexpr int kSegPlanes = (\d+);", src).group(1))


def test_segment_plans_stay_inside_their_bounds(plans):
    planes = _seg_planes()
    taken = 0
    for sms, nl, H, mc, P, L, *_ in plans:
        if P == 0:
            continue
        taken += 1
        pairs = nl * H
        assert pairs <= 4 and mc >= 12, (sms, nl, H, mc)
        assert 3 * pairs * (P - 1) <= planes, (sms, nl, H, mc, P)   # workspace planes
        assert 16 * pairs * (P - 1) <= sms, (sms, nl, H, mc, P)     # pass A: one wave
        assert L >= 4 and P >= 2, (mc, P, L)                        # segments of 4+ chunks
        assert (P - 1) * L < mc <= P * L, (mc, P, L)                # every chunk, no empty segment
    assert taken > 0


def test_known_plans(plans):
    by = {(s, nl, H, mc): (P, L) for s, nl, H, mc, P, L, *_ in plans}
    assert by[(152, 1, 2, 256)] == (5, 52)    # 1 x 16384, H = 2: five segments of 52 chunks
    assert by[(152, 1, 6, 256)][0] == 0       # 6 pairs: the fused launch or the plain scan
    assert by[(152, 1, 1, 11)][0] == 0        # too short to cut


def test_value_row_split(plans):
    # 16 value rows per CTA while the walks of 16 fill at most two waves, 64 while
    # the walks of 64 fit one wave, else 128; with a wave of token-by-token pairs
    # beside the scan, 128 in place of 64
    for sms, nl, H, mc, P, L, groups, groups_beside in plans:
        pairs = nl * H
        want = 1 if pairs * 8 <= 2 * sms else (4 if pairs * 2 <= sms else 8)
        assert groups == want, (sms, nl, H, groups)
        assert groups_beside == (1 if want == 1 else 8), (sms, nl, H, groups_beside)
    assert any(g == 4 for *_, g, _ in plans) and any(g == 8 for *_, g, _ in plans)
