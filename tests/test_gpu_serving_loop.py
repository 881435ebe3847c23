"""A small serving loop on the GPU driven by the host block manager:
prefill through pa_cache_update, sequences forked from a shared prefix,
then decode steps with pa_decode, every step checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_300_gb300 as pa
from tests.gpu_util import assert_close, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pa.load()


def test_block_manager_prefill_fork_decode():
    from paged_kv_cache_300_gb300.blocks import BlockManager
    nb, bs, mb, hq, hkv, d = 64, 16, 16, 8, 2, 128
    g = torch.Generator().manual_seed(77)
    rnd = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)
    kc = rnd(nb, bs, hkv, d).cuda()
    vc = rnd(nb, bs, hkv, d).cuda()
    bm = BlockManager(nb, bs, mb)
    # prefill sequence 0 (40 tokens) through the cache update
    bm.add(0, 40)
    t, _ = bm.tables([0])
    kch, vch = rnd(40, hkv, d), rnd(40, hkv, d)
    pa.pa_cache_update(kch.cuda(), vch.cuda(), torch.tensor([0, 40], dtype=torch.int32).cuda(),
                       torch.tensor([0], dtype=torch.int32).cuda(), t.cuda(), kc, vc)
    # sequences 1, 2 share its first two full blocks (32 tokens) and add 3 / 9 own tokens
    for s, extra in ((1, 3), (2, 9)):
        bm.fork(0, s, 32)
        prefix = bm.length(s)
        bm.append(s, extra)
        t, _ = bm.tables([s])
        pa.pa_cache_update(rnd(extra, hkv, d).cuda(), rnd(extra, hkv, d).cuda(),
                           torch.tensor([0, extra], dtype=torch.int32).cuda(),
                           torch.tensor([prefix], dtype=torch.int32).cuda(), t.cuda(), kc, vc)
    torch.cuda.synchronize()
    seqs = [0, 1, 2]
    for step in range(5):
        for s in seqs:
            bm.append(s, 1)   # room for this step's token
        table, lengths = bm.tables(seqs)
        sl = (lengths - 1).to(torch.int32)  # cached tokens before the new one
        q, kn, vn = rnd(3, hq, d), rnd(3, hkv, d), rnd(3, hkv, d)
        rk, rv = bits(kc).copy(), bits(vc).copy()
        out = pa.pa_decode(q.cuda(), kc, vc, table.cuda(), sl.cuda(), kn.cuda(), vn.cuda())
        torch.cuda.synchronize()
        ref = oracle.decode(bits(q), rk, rv, table.numpy(), sl.numpy(), bits(kn), bits(vn))
        assert_close(out, ref, torch.bfloat16, f"step {step}")
        assert np.array_equal(bits(kc), rk) and np.array_equal(bits(vc), rv)
    # the shared blocks are still shared and nothing leaked
    shared = table[0, :2].tolist()
    assert table[1, :2].tolist() == shared and table[2, :2].tolist() == shared
    assert [bm.refcount(b) for b in shared] == [3, 3]
    for s in seqs:
        bm.free(s)
    assert bm.num_free() == nb


@pytest.mark.parametrize("mode", ["stream", "graph"])
def test_back_to_back_steps_each_reading_the_last_append(mode):
    """K decode steps launched back to back with no host synchronisation (on
    one stream, or captured as one CUDA graph as the benchmark runs them),
    step t attending over the token step t-1 appended and sharing one
    workspace.  Each launch allows programmatic dependence, so a step's
    start-up overlaps the previous step; every output and both pools must
    still equal the oracle run step by step."""
    b, hq, hkv, d, bs, steps = 24, 32, 8, 128, 16, 6
    g = torch.Generator().manual_seed(4242)
    lens = torch.randint(200, 1500, (b,), generator=g)
    mbps = (int(lens.max()) + steps + bs - 1) // bs
    need = [(int(n) + steps + bs - 1) // bs for n in lens]
    nb = sum(need) + 8
    perm = torch.randperm(nb, generator=g)
    table = torch.full((b, mbps), -1, dtype=torch.int32)
    o = 0
    for s in range(b):
        table[s, :need[s]] = perm[o:o + need[s]]
        o += need[s]
    rnd = lambda *sh: torch.randn(*sh, generator=g).to(torch.bfloat16)
    kc0, vc0 = rnd(nb, bs, hkv, d), rnd(nb, bs, hkv, d)
    qs = [rnd(b, hq, d) for _ in range(steps)]
    kns = [rnd(b, hkv, d) for _ in range(steps)]
    vns = [rnd(b, hkv, d) for _ in range(steps)]
    sls = [(lens + t).to(torch.int32) for t in range(steps)]
    dev = "cuda"
    kc, vc = kc0.to(dev), vc0.to(dev)
    tab = table.to(dev)
    dq = [x.to(dev) for x in qs]
    dkn = [x.to(dev) for x in kns]
    dvn = [x.to(dev) for x in vns]
    dsl = [x.to(dev) for x in sls]
    outs = [torch.empty(b, hq, d, dtype=torch.bfloat16, device=dev) for _ in range(steps)]
    ws = torch.zeros(pa.pa_decode_workspace_size(b, hq, hkv, d, bs), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def run_all():
        for t in range(steps):
            pa.pa_decode(dq[t], kc, vc, tab, dsl[t], dkn[t], dvn[t], outs[t], workspace=ws,
                         dev_err=err)

    if mode == "graph":
        run_all()  # first calls outside capture (plan and descriptor set-up)
        torch.cuda.synchronize()
        kc.copy_(kc0)
        vc.copy_(vc0)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run_all()
        torch.cuda.synchronize()
        kc.copy_(kc0)
        vc.copy_(vc0)
        for x in outs:
            x.zero_()
        torch.cuda.synchronize()
        graph.replay()
    else:
        run_all()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rk, rv = bits(kc0).copy(), bits(vc0).copy()
    for t in range(steps):
        ref = oracle.decode(bits(qs[t]), rk, rv, table.numpy(), sls[t].numpy(), bits(kns[t]),
                            bits(vns[t]))
        assert_close(outs[t], ref, torch.bfloat16, f"{mode} step {t}")
    assert np.array_equal(bits(kc), rk) and np.array_equal(bits(vc), rv)
