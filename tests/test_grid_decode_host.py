"""The standard kernel's work-item grid on the CPU: the host's grid set-up
(make_grid_spec) and the kernel's item decoding (decode_item, multiply-shift
divisions) compiled from the same header into a host program, which walks
every item of 400 grid shapes -- MHA and GQA with even and odd group sizes,
odd query-block counts, head counts that leave a narrower last strip of 8,
both item orders -- and checks that every (batch, head, query block) is
visited exactly once, that the two slots of an item share its KV head (MHA:
consecutive query blocks of one head; GQA: two heads of one KV group at one
query block), and that the longest-first order never raises the query block."""
import os
import shutil
import subprocess

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "attention_variant_gb300", "csrc")
INCLUDE = os.path.join(os.path.dirname(CSRC), "..", "include")

PROGRAM = r"""
#include <cstdio>
#include <vector>
#include "common.cuh"

using namespace fl;
static long bad = 0, items = 0;

static void fail(const char *what, int B, int Hq, int Hk, int nq, int lpt, long long L) {
    if (bad < 10)
        std::printf("%s: B=%d Hq=%d Hk=%d nq=%d lpt=%d item %lld\n", what, B, Hq, Hk, nq, lpt, L);
    ++bad;
}

static void check(int B, int Hq, int Hk, int nq, int lpt) {
    GridSpec g{};
    if (!make_grid_spec(B, Hq, Hk, nq, lpt != 0, g)) { fail("refused", B, Hq, Hk, nq, lpt, -1); return; }
    const int G = Hq / Hk;
    std::vector<int> seen(size_t(B) * Hq * nq, 0);
    int last_qb = 1 << 30;
    for (long long L = 0; L < g.n_items; ++L, ++items) {
        const Item it = decode_item(g, L);
        if (it.b < 0 || it.b >= B || it.kvh < 0 || it.kvh >= Hk) { fail("out of range", B, Hq, Hk, nq, lpt, L); continue; }
        if (!it.valid[0]) fail("slot 0 absent", B, Hq, Hk, nq, lpt, L);
        for (int t = 0; t < 2; ++t) {
            if (!it.valid[t]) continue;
            const int h = it.h[t], qb = it.qb[t];
            if (h < 0 || h >= Hq || qb < 0 || qb >= nq || h / G != it.kvh) { fail("bad slot", B, Hq, Hk, nq, lpt, L); continue; }
            ++seen[(size_t(it.b) * Hq + h) * nq + qb];
        }
        if (it.valid[0] && it.valid[1]) {
            if (G == 1 && !(it.h[0] == it.h[1] && it.qb[1] == it.qb[0] + 1)) fail("MHA slots", B, Hq, Hk, nq, lpt, L);
            if (G >= 2 && !(it.qb[0] == it.qb[1] && it.h[1] == it.h[0] + 1)) fail("GQA slots", B, Hq, Hk, nq, lpt, L);
        }
        if (lpt) {
            if (it.qb[0] > last_qb) fail("LPT order", B, Hq, Hk, nq, lpt, L);
            last_qb = it.qb[0];
        }
    }
    for (size_t x = 0; x < seen.size(); ++x)
        if (seen[x] != 1) { fail("visits != 1", B, Hq, Hk, nq, lpt, (long long)x); break; }
}

int main() {
    const int heads[10][2] = {{1, 1}, {4, 4}, {6, 6}, {16, 16}, {5, 5}, {8, 2}, {6, 2}, {3, 1}, {16, 2}, {12, 4}};
    int configs = 0;
    for (int B : {1, 2, 3, 5})
        for (const auto &hh : heads)
            for (int nq : {1, 2, 3, 16, 17})
                for (int lpt = 0; lpt < 2; ++lpt, ++configs)
                    check(B, hh[0], hh[1], nq, lpt);
    std::printf("configs %d items %ld bad %ld\n", configs, items, bad);
    return bad == 0 ? 0 : 1;
}
"""


def test_work_item_grid_visits_every_tile_once(tmp_path):
    nvcc = shutil.which(os.environ.get("NVCC", "nvcc"))
    if nvcc is None:
        pytest.skip("nvcc is not available")
    src = tmp_path / "grid_check.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "grid_check"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O1",
                    "-I", CSRC, "-I", INCLUDE, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "configs 400" in r.stdout and "bad 0" in r.stdout, r.stdout
