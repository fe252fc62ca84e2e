"""CPU checks on the CUDA sources: forms this library must never contain.

- A TMA load with cluster multicast (cp.async.bulk ... .multicast::cluster): the library is
  loaded by every rank of a multi-GPU run, and no such load may appear in code that can run
  on several GPUs.
- The batched memcpy entry points of the runtime and driver APIs (the 2-D and 3-D batch
  forms): one cudaMemcpyAsync per copy, or a gather kernel, is used instead.
"""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "mla_latent_kv_79_b300", "csrc")


def _sources():
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            yield name, open(os.path.join(CSRC, name)).read()


def _statements(text):
    """asm strings joined across adjacent string literals, one instruction per ';'."""
    joined = re.sub(r'"\s*\n\s*"', "", text)
    return joined.split(";")


def test_no_multicast_bulk_copy():
    bad = []
    for name, text in _sources():
        for stmt in _statements(text):
            if "cp.async.bulk" in stmt and "multicast::cluster" in stmt:
                bad.append((name, stmt.strip()[:120]))
    assert not bad, bad


def test_no_batched_memcpy():
    pat = re.compile("cu(da)?Memcpy(3D)?" + "Batch" + "Async")
    for root in (CSRC, os.path.join(ROOT, "include")):
        for name in os.listdir(root):
            path = os.path.join(root, name)
            if os.path.isfile(path):
                assert not pat.search(open(path, errors="ignore").read()), path


def test_the_check_sees_a_planted_multicast_load():
    planted = ('asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"\n'
               '             ".multicast::cluster [%0], [%1, {%2, %3}], [%4], %5;" ::);')
    assert any("cp.async.bulk" in s and "multicast::cluster" in s for s in _statements(planted))
