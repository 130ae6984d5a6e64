"""The block manager driving the GPU cache: a multi-step generation -- prefill, decode
steps, a fork (shared prefix) followed by copy on write, a finished sequence whose blocks
are reused -- with every decode checked against the fp64 oracle over each sequence's
logical K/V.  Also pa_copy_blocks on its own, byte for byte."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import assert_close

import paged_decode_attention_reshape_gb300 as pa

pytestmark = pytest.mark.gpu
B = 16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_decode_attention_reshape_gb300 import _build
    _build.build()
    pa.lib()
    torch.cuda.set_device(0)


class Engine:
    """Sequences on a paged bf16 cache, bookkept by the library's block manager."""

    def __init__(self, NB=48, NS=8, MB=12, Hq=32, Hkv=8, D=128, seed=0):
        self.m = pa.BlockManager(NB, NS, MB)
        self.Hq, self.Hkv, self.D, self.MB = Hq, Hkv, D, MB
        self.kc = torch.full((NB, Hkv, B, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        self.vc = torch.full_like(self.kc, float("nan"))
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.logical = {}                       # seq -> (K, V) [L, Hkv, D] bf16 on the host
        self.g = torch.Generator().manual_seed(seed)
        self.copies = 0

    def append(self, s, n):
        K = torch.randn(n, self.Hkv, self.D, generator=self.g).to(torch.bfloat16)
        V = torch.randn(n, self.Hkv, self.D, generator=self.g).to(torch.bfloat16)
        slots, cp = self.m.append(s, n)
        if cp is not None:                      # copy on write before the token lands
            pa.pa_copy_blocks(self.kc, self.vc, torch.tensor([cp], dtype=torch.int64, device="cuda"), self.err)
            self.copies += 1
        pa.pa_reshape_and_cache(K.cuda(), V.cuda(), self.kc, self.vc, torch.from_numpy(slots).cuda(),
                                pa.PA_KV_AUTO, None, None, self.err)
        k0, v0 = self.logical.get(s, (K[:0], V[:0]))
        self.logical[s] = (torch.cat([k0, K]), torch.cat([v0, V]))

    def fork(self, src, dst):
        self.m.fork(src, dst)
        self.logical[dst] = tuple(t.clone() for t in self.logical[src])

    def free(self, s):
        self.m.free(s)
        self.logical.pop(s, None)

    def check(self, seqs, what):
        bt, sl = self.m.export(seqs)
        assert list(sl) == [self.logical[s][0].shape[0] for s in seqs]
        q = torch.randn(len(seqs), self.Hq, self.D, generator=self.g).to(torch.bfloat16)
        ref = np.stack([oracle.dense_decode(q[i].double().numpy(), self.logical[s][0].double().numpy(),
                                            self.logical[s][1].double().numpy(), self.D ** -0.5)
                        for i, s in enumerate(seqs)])
        btd, sld, qd = torch.from_numpy(bt).cuda(), torch.from_numpy(sl).cuda(), q.cuda()
        ws = torch.zeros(8 << 20, dtype=torch.uint8, device="cuda")
        for P in (-1, 32, -2):
            out = torch.empty_like(qd)
            pa.pa_decode_ex(out, qd, self.kc, self.vc, btd, sld, self.D ** -0.5, self.Hkv, None, None, P, ws,
                            self.err)
            assert pa.pa_check_device_error(self.err) == (0, 0)
            assert_close(out.double().cpu().numpy(), ref, "%s, partition %d" % (what, P))


def test_generation_with_fork_copy_on_write_and_reuse():
    e = Engine()
    for s, L in enumerate([20, 37, 5, 60]):            # prefill
        e.append(s, L)
    e.check([0, 1, 2, 3], "after prefill")
    for step in range(5):                              # decode steps
        for s in range(4):
            e.append(s, 1)
        e.check([0, 1, 2, 3], "decode step %d" % step)
    e.fork(0, 4)                                       # seq 0 has 25 tokens: its last block is shared, partial
    e.append(4, 1)                                     # -> copy on write for the fork
    e.append(0, 1)                                     # the block is seq 0's alone again: no copy
    assert e.copies == 1
    e.check([0, 1, 2, 3, 4], "after fork")
    free_before = e.m.num_free()
    e.free(1)                                          # seq 1 finishes; its blocks are reused
    assert e.m.num_free() == free_before + 3
    e.append(5, 40)
    e.fork(3, 6)
    for step in range(3):
        for s in (0, 2, 3, 4, 5, 6):
            e.append(s, 1 + step)
        e.check([0, 2, 3, 4, 5, 6], "after reuse, step %d" % step)
    assert e.copies == 2                               # the second fork's first append copied too


@pytest.mark.parametrize("layout,dt", [("hnd", torch.bfloat16), ("nhd", torch.uint8), ("hnd", torch.float32)])
def test_copy_blocks_bytes(layout, dt):
    NB, Hkv, D = 20, 4, 128
    shape = (NB, B, Hkv, D) if layout == "nhd" else (NB, Hkv, B, D)
    g = torch.Generator().manual_seed(3)
    kb = torch.randint(0, 255, shape, generator=g, dtype=torch.uint8)
    vb = torch.randint(0, 255, shape, generator=g, dtype=torch.uint8)
    if dt != torch.uint8:
        kb = torch.randn(shape, generator=g).to(dt)
        vb = torch.randn(shape, generator=g).to(dt)
    k, v = kb.cuda(), vb.cuda()
    view = (lambda t: t.permute(0, 2, 1, 3)) if layout == "nhd" else (lambda t: t)
    pairs = torch.tensor([[3, 7], [0, 19], [12, 5]], dtype=torch.int64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(view(k), view(v), pairs.cuda(), err)
    assert pa.pa_check_device_error(err) == (0, 0)
    ek, ev = kb.clone(), vb.clone()
    for a, b in pairs.tolist():
        ek[b], ev[b] = kb[a], vb[a]
    assert torch.equal(k.cpu().view(torch.uint8), ek.view(torch.uint8))
    assert torch.equal(v.cpu().view(torch.uint8), ev.view(torch.uint8))
    pa.pa_copy_blocks(view(k), view(v), torch.tensor([[1, NB]], dtype=torch.int64, device="cuda"), err)
    rc, bits = pa.pa_check_device_error(err)
    assert rc == -6 and bits & pa.PA_DEVERR_BLOCK_RANGE
