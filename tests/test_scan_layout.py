"""Host logic of the state launches' CTA decomposition (no GPU needed).

Every state launch numbers its CTAs in groups of one (sequence rank, state
head); scan_cta maps a CTA index to (rank, head, segment, tile, role) and
scan_ctas_per_group gives the group size the host launches.  For the
chunk-parallel pass the first launch replays segment 0 beside the
transitions of segments 1 .. P - 2 (two column tiles per transition), and the
replay launch covers segments 1 .. P - 1.  This compiles a small host program
against the library's internal header and checks, for every mode, segment
count, tile count, head count and sequence count, that the CTAs cover exactly
those (sequence, head, segment, tile) units, each once.
"""
import os
import subprocess

import pytest

from gated_deltanet_prefill_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <cstdio>
#include <set>
#include <tuple>
#include "gdn2_internal.cuh"
using namespace gdn2;

int main() {
    int bad = 0, cases = 0;
    for (int mode = 0; mode < 3; ++mode)
        for (int P = mode == 0 ? 1 : 2; P <= (mode == 0 ? 1 : 17); ++P)
            for (int rt = 1; rt <= 2; ++rt)
                for (int HV : {1, 3, 4})
                    for (int N : {1, 2, 5}) {
                        ++cases;
                        const int per = scan_ctas_per_group(mode, P, rt);
                        std::set<std::tuple<int, int, int, int, int>> seen;
                        for (int b = 0; b < N * HV * per; ++b) {
                            const ScanCta c = scan_cta(b, mode, P, HV, rt);
                            const int ntile = c.trans ? 2 * rt : rt;
                            bool ok = c.rank >= 0 && c.rank < N && c.hv >= 0 && c.hv < HV && c.tile >= 0 &&
                                      c.tile < ntile && b / per == c.rank * HV + c.hv;
                            if (mode == 0) ok = ok && c.seg == 0 && !c.trans;
                            if (mode == 1) ok = ok && (c.trans ? c.seg >= 1 && c.seg <= P - 2 : c.seg == 0);
                            if (mode == 2) ok = ok && !c.trans && c.seg >= 1 && c.seg <= P - 1;
                            ok = ok && seen.insert(std::make_tuple(c.rank, c.hv, c.seg, c.tile, int(c.trans))).second;
                            if (!ok) {
                                if (bad < 10)
                                    printf("mode %d P %d rt %d HV %d N %d b %d -> rank %d hv %d seg %d tile %d trans %d\n",
                                           mode, P, rt, HV, N, b, c.rank, c.hv, c.seg, c.tile, int(c.trans));
                                ++bad;
                            }
                        }
                        const size_t units = mode == 0 ? rt : mode == 1 ? rt + 2 * rt * (P - 2) : rt * (P - 1);
                        if (seen.size() != static_cast<size_t>(N) * HV * units) ++bad;
                    }
    printf("%s %d cases, %d bad\n", bad ? "FAIL" : "OK", cases, bad);
    return bad != 0;
}
"""


def test_scan_cta_covers_every_unit_once(tmp_path):
    nvcc = gbuild.nvcc()
    src = tmp_path / "scan_layout.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "scan_layout"
    csrc = os.path.join(ROOT, "gated_deltanet_prefill_gb300", "csrc")
    cmd = [nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-I", csrc, "-I",
           os.path.join(ROOT, "include"), str(src), "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        pytest.fail("nvcc failed:\n" + r.stderr[-2000:])
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.startswith("OK"), out.stdout[-2000:]
