"""The long-sequence split planner of the tensor-core prefill (plan_split_search,
pass1_entries, pass2_entries in csrc/kda_chunk_tc.cu), compiled for the host
and run on the CPU (nothing launches).  For every planned sequence the
segments tile its tokens in 64-token steps; segment 0 runs once from the
caller's state in pass 1 and hands its final state to slot base + 1; every
inner segment runs twice in pass 1 (S~ from zero into slot E + base + q, M
from the identity with v = 0 into slot 2E + base + q, neither writing
outputs) and again in pass 2 from slot base + q; the last segment writes the
caller's final state.  The long single-sequence workload's plan is pinned
(a longer first segment), and a batch that fills the GPU is not split."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "linear_attention_layer_gb300", "csrc")
USER, ZERO, IDENTITY, NONE = -3, -1, -2, -1
ZERO_V, NO_OUT = 1, 2


@pytest.fixture(scope="module")
def planner(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("no nvcc")
    exe = str(tmp_path_factory.mktemp("plan") / "plan_driver")
    src = os.path.join(ROOT, "tests", "host", "plan_driver.cu")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O1",
                    "-I", CSRC, "-I", os.path.join(ROOT, "include"), src, "-o", exe],
                   check=True, capture_output=True)
    return exe


def _plan(exe, lens, H, sms=152):
    inp = f"{H} {sms}\n" + " ".join(map(str, lens)) + "\n"
    out = subprocess.run([exe], input=inp, capture_output=True, text=True, check=True).stdout
    plan, seqs, p1, p2 = None, {}, [], []
    for line in out.strip().split("\n"):
        f = line.split()
        if f[0] == "plan":
            plan = dict(zip(("use", "seg0", "seg", "s0_at", "E"), map(int, f[1:])))
        elif f[0] == "seq":
            seqs[int(f[1])] = (int(f[2]), int(f[3]))
        else:
            (p1 if f[0] == "p1" else p2).append(tuple(map(int, f[1:])))
    return plan, seqs, p1, p2


def _check(lens, plan, seqs, p1, p2):
    cu = [0]
    for l in lens:
        cu.append(cu[-1] + l)
    E = plan["E"]
    assert plan["seg0"] % 64 == 0 and plan["seg"] % 64 == 0 and plan["seg0"] >= plan["seg"]
    assert sum(k for k, _ in seqs.values()) == E
    for n, (k, b) in seqs.items():
        mine1 = [e for e in p1 if e[0] == n]
        mine2 = sorted((e for e in p2 if e[0] == n), key=lambda e: e[1])
        if k == 1:  # unsplit: one pass-2 run over the whole sequence from slot base
            assert mine1 == [] and mine2 == [(n, cu[n], cu[n + 1], b, USER, 0)]
            continue
        first = [e for e in mine1 if e[3] == USER]
        assert first == [(n, cu[n], cu[n] + plan["seg0"], USER, b + 1, 0)]
        inner = [e for e in mine1 if e[3] != USER]
        assert len(inner) == 2 * (k - 2) and len(mine2) == k - 1
        bounds = [cu[n]] + [cu[n] + plan["seg0"] + q * plan["seg"] for q in range(k - 1)] + [cu[n + 1]]
        for q in range(1, k):
            tb, te = bounds[q], bounds[q + 1]
            assert te > tb and (q == k - 1 or te - tb == plan["seg"])
            assert mine2[q - 1] == (n, tb, te, b + q, USER if q == k - 1 else NONE, 0)
            if q < k - 1:
                assert (n, tb, te, ZERO, E + b + q, NO_OUT) in inner
                assert (n, tb, te, IDENTITY, 2 * E + b + q, ZERO_V | NO_OUT) in inner


def test_long_sequence_plan(planner):
    lens = [65536]
    plan, seqs, p1, p2 = _plan(planner, lens, 32)
    assert plan["use"] == 1
    assert (plan["seg0"] // 64, plan["seg"] // 64) == (342, 171)  # segment 0 twice the rest
    assert seqs[0][0] == 5
    _check(lens, plan, seqs, p1, p2)
    # segment 0's entries sit where no CTA holding one gets a second pass-1 unit
    units = [e for e in p1 for _ in range(32)]
    heavy = {u % 152 for u, e in enumerate(units) if e[3] == USER}
    light2 = {u % 152 for u in range(152, len(units))}
    assert not heavy & light2


@pytest.mark.parametrize("lens,H", [([4096] * 4, 16), ([3000, 1100], 2), ([3000, 700, 2], 2),
                                    ([20000, 27000, 34000], 8)])
def test_split_plans_tile_every_sequence(planner, lens, H):
    plan, seqs, p1, p2 = _plan(planner, lens, H)
    assert plan["use"] == 1
    _check(lens, plan, seqs, p1, p2)


def test_a_batch_that_fills_the_gpu_is_not_split(planner):
    plan, _, _, _ = _plan(planner, [2048] * 64, 32)
    assert plan["use"] == 0
