"""Host logic of offload mode (no GPU): the HBM slot placement of
csrc/slot_cache.h, compiled with the host compiler into a small driver.

Policy (per batch of distinct experts of one layer): hits keep their slot and
are refreshed first; each miss then takes the lowest empty slot, else the
least recently used slot that this batch does not use."""

import os
import random
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "nvfp4_mixture_experts_counting_gb300", "csrc")

DRIVER = r"""
#include <cstdio>
#include "slot_cache.h"
// stdin: n_slots n_layers n_experts n_batches, then per batch: layer n e_1 .. e_n
// stdout per batch: slot miss pairs; at the end hits and misses per layer
int main() {
  int ns, nl, ne, nb;
  if (std::scanf("%d %d %d %d", &ns, &nl, &ne, &nb) != 4) return 1;
  ftmoe::SlotCache c;
  c.reset(ns, nl, ne);
  for (int b = 0; b < nb; ++b) {
    int layer, n;
    if (std::scanf("%d %d", &layer, &n) != 2) return 1;
    std::vector<int> ex(n);
    for (int i = 0; i < n; ++i)
      if (std::scanf("%d", &ex[i]) != 1) return 1;
    auto pl = c.place(layer, ex.data(), n);
    for (auto& p : pl) std::printf("%d %d ", p.slot, p.miss ? 1 : 0);
    std::printf("\n");
  }
  for (int l = 0; l < nl; ++l) std::printf("%lld %lld\n", (long long)c.hits(l), (long long)c.misses(l));
  return 0;
}
"""


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("slot_cache")
    src, exe = d / "drv.cpp", d / "drv"
    src.write_text(DRIVER)
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    return str(exe)


def run(driver, ns, nl, ne, batches):
    inp = f"{ns} {nl} {ne} {len(batches)}\n" + "".join(
        f"{layer} {len(ex)} {' '.join(map(str, ex))}\n" for layer, ex in batches)
    out = subprocess.run([driver], input=inp, capture_output=True, text=True, check=True).stdout.split("\n")
    placements = []
    for b, (layer, ex) in enumerate(batches):
        v = list(map(int, out[b].split()))
        placements.append([(v[2 * i], bool(v[2 * i + 1])) for i in range(len(ex))])
    counts = [tuple(map(int, out[len(batches) + l].split())) for l in range(nl)]
    return placements, counts


def model(ns, nl, ne, batches):
    """The policy, step by step: slot -> (layer, expert, last use)."""
    occ = [None] * ns
    clock = 0
    hits = [0] * nl
    misses = [0] * nl
    res = []
    for layer, ex in batches:
        start = clock + 1
        pl = [None] * len(ex)
        where = {(o[0], o[1]): s for s, o in enumerate(occ) if o is not None}
        for i, e in enumerate(ex):
            s = where.get((layer, e))
            if s is not None:
                clock += 1
                occ[s] = (layer, e, clock)
                pl[i] = (s, False)
                hits[layer] += 1
        for i, e in enumerate(ex):
            if pl[i] is not None:
                continue
            empty = [s for s in range(ns) if occ[s] is None]
            if empty:
                v = empty[0]
            else:
                v = min((s for s in range(ns) if occ[s][2] < start), key=lambda s: occ[s][2])
            clock += 1
            occ[v] = (layer, e, clock)
            pl[i] = (v, True)
            misses[layer] += 1
        res.append(pl)
    return res, list(zip(hits, misses))


def test_hand_worked_two_slots(driver):
    # A, B fill slots 0 and 1; C evicts A (older); A then evicts B
    pl, counts = run(driver, 2, 1, 4, [(0, [0, 1]), (0, [2]), (0, [0])])
    assert pl == [[(0, True), (1, True)], [(0, True)], [(1, True)]]
    assert counts == [(0, 4)]


def test_hits_keep_their_slot_and_a_batch_never_evicts_itself(driver):
    # slots 0..2 hold 0, 1, 2; the batch [2, 5, 6] keeps 2 and evicts 0 and 1
    pl, counts = run(driver, 3, 1, 8, [(0, [0, 1, 2]), (0, [2, 5, 6])])
    assert pl[1][0] == (2, False)
    assert sorted(s for s, m in pl[1][1:]) == [0, 1] and all(m for _, m in pl[1][1:])
    assert counts == [(1, 5)]


def test_layers_share_the_pool(driver):
    pl, counts = run(driver, 2, 2, 4, [(0, [1]), (1, [1]), (0, [1]), (1, [2])])
    assert pl[2] == [(0, False)]          # layer 0's expert 1 is still in slot 0
    assert pl[3] == [(1, True)]           # layer 1's expert 1 (slot 1) is the older one
    assert counts == [(1, 1), (0, 2)]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_batches_match_the_policy(driver, seed):
    rng = random.Random(seed)
    ns, nl, ne = 7, 3, 20
    batches = []
    for _ in range(60):
        layer = rng.randrange(nl)
        batches.append((layer, rng.sample(range(ne), rng.randint(1, ns))))
    got = run(driver, ns, nl, ne, batches)
    assert got == model(ns, nl, ne, batches)
    # within a batch every expert has its own slot
    for pl in got[0]:
        assert len({s for s, _ in pl}) == len(pl)
