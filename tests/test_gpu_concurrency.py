"""Concurrent use: one-shot digests from several host threads on their own streams, and
two streaming hashers interleaved on two streams; every result equals the oracle's."""

import threading

import pytest
import torch

import oracle
from blake3_merkle_tree_gb300 import binding, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from blake3_merkle_tree_gb300 import build

    build.build()
    binding.library()
    yield
    assert binding.blake3_device_status() == 0


def test_threads_on_their_own_streams():
    lengths = [1025, (3 << 20) + 7, 64 << 20, (9 << 20) + 777, 5000, (33 << 20) + 1]
    hosts = [workloads.uniform_bytes(5000 + i, n) for i, n in enumerate(lengths)]
    keys = [workloads.key_bytes(5100 + i) for i in range(len(lengths))]
    devs = [h.cuda() for h in hosts]
    results = [None] * len(lengths)
    errors = []

    def work(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                outs = []
                for _ in range(4):
                    if i % 2:
                        outs.append(binding.blake3_keyed_hash(devs[i], keys[i]))
                    else:
                        outs.append(binding.blake3_hash(devs[i]))
            s.synchronize()
            results[i] = {bytes(o.cpu().numpy()) for o in outs}
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(lengths))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, h in enumerate(hosts):
        ref = oracle.keyed_hash(h, keys[i]) if i % 2 else oracle.hash(h)
        assert results[i] == {ref}, i


def test_two_hashers_interleaved_on_two_streams():
    n = (48 << 20) + 123
    a_host = workloads.uniform_bytes(5200, n)
    b_host = workloads.uniform_bytes(5201, n)
    a, b = a_host.cuda(), b_host.cuda()
    key = workloads.key_bytes(5202)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    ha, hb = binding.Hasher(key), binding.Hasher()
    cuts = [0, 777, 1 << 20, (5 << 20) + 3, (20 << 20) + 1, (40 << 20) + 9, n]
    for x, y in zip(cuts[:-1], cuts[1:]):
        ha.update(a[x:y], stream=sa)
        hb.update(b[x:y], stream=sb)
    oa = ha.finalize(stream=sa)
    ob = hb.finalize(stream=sb)
    sa.synchronize()
    sb.synchronize()
    assert bytes(oa.cpu().numpy()) == oracle.keyed_hash(a_host, key)
    assert bytes(ob.cpu().numpy()) == oracle.hash(b_host)
