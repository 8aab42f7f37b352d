"""Host-side tagging of the dynamic schedule's launches (sched_ticket.h),
compiled on its own with the host C++ compiler: every launch gets a slot and a
nonzero generation, slots go round-robin unless pinned, and generations of
launches in flight together never coincide (CPU only)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "attention_forward_14_gb300", "csrc")

DRIVER = r"""
#include <cstdio>
#include <cstdlib>
#include "sched_ticket.h"
using namespace attn;
int main(int argc, char **argv) {
    // argv: first launch index, count, pinned slot
    const unsigned long long n0 = strtoull(argv[1], nullptr, 10), cnt = strtoull(argv[2], nullptr, 10);
    const int pinned = atoi(argv[3]);
    for (unsigned long long i = 0; i < cnt; ++i) {
        const SchedTicket t = sched_ticket(n0 + i, pinned);
        printf("%d %u\n", t.slot, t.gen);
    }
    return 0;
}
"""


@pytest.fixture(scope="module")
def ticket(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("ticket")
    src, exe = d / "t.cpp", d / "t"
    src.write_text(DRIVER)
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)

    def run(n0, cnt, pinned=-1):
        out = subprocess.run([str(exe), str(n0), str(cnt), str(pinned)], check=True, capture_output=True, text=True)
        return [tuple(int(x) for x in ln.split()) for ln in out.stdout.splitlines()]
    return run


def test_slots_round_robin_and_generations_distinct(ticket):
    t = ticket(0, 1000)
    assert [s for s, _ in t] == [i % 256 for i in range(1000)]
    gens = [g for _, g in t]
    assert 0 not in gens and len(set(gens)) == len(gens)
    # the 256 launches that share a slot round by round carry distinct tags
    assert len({g for s, g in t if s == 5}) == len([1 for s, _ in t if s == 5])


def test_generation_never_zero_across_the_wrap(ticket):
    n0 = (1 << 32) - 600
    t = ticket(n0, 1200)
    gens = [g for _, g in t]
    assert 0 not in gens
    assert all(0 < g < (1 << 32) for g in gens)
    assert len(set(gens)) == len(gens)  # 1200 consecutive launches: no repeat
    assert [s for s, _ in t] == [(n0 + i) % 256 for i in range(1200)]


def test_pinned_slot_is_honoured_and_bad_pins_ignored(ticket):
    assert {s for s, _ in ticket(10, 50, pinned=7)} == {7}
    assert [s for s, _ in ticket(10, 3, pinned=256)] == [10, 11, 12]
    gens = [g for _, g in ticket(10, 50, pinned=7)]
    assert len(set(gens)) == 50
