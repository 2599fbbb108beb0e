"""Back-to-back launches on one stream and concurrent launches on two.

Every GEMM kernel of the library is launched with programmatic dependent
launch: its CTAs may start on SMs the previous kernel has left and must not
touch global memory before that kernel has completed.  These tests chain
products whose each input is the previous output (read after write), in
ping-pong buffers so that each launch overwrites what the one before it read
(write after read), with no synchronisation between launches.  The same
chain run with a device synchronisation after every launch is the
reference: the library's results are deterministic, so the two must agree
bit for bit, and a launch that read or wrote too early would break that.

The skinny split-K kernel also runs on two streams at once: its launch has no
co-residency requirement (no CTA waits for another), so two such grids
sharing the SMs must both finish, each with the results it gives alone.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from tiled_fp16_gemm_gb300 import workloads as W  # noqa: E402


@pytest.fixture(scope="module")
def tg():
    from tiled_fp16_gemm_gb300 import build
    build.build()
    import tiled_fp16_gemm_gb300 as t
    return t


def _weights(n, k, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(k, n, generator=g) / np.sqrt(k)).half().cuda()


def _run_chain(step, bufs, steps, sync_each):
    for i in range(steps):
        step(i, bufs)
        if sync_each:
            torch.cuda.synchronize()
    torch.cuda.synchronize()


def _same(tg, step, make_bufs, steps=8):
    ref = make_bufs()
    _run_chain(step, ref, steps, sync_each=True)
    tg.sync_status()
    got = make_bufs()
    _run_chain(step, got, steps, sync_each=False)
    tg.sync_status()
    for k in ref:
        assert torch.isfinite(ref[k].float()).all(), k
        assert torch.equal(ref[k], got[k]), f"buffer {k} differs from the synchronised chain"


# (name, M, K=N, forced configuration): the pair kernel, the one-CTA kernel
# with both tile widths, and the skinny kernel
DENSE = [("pair", 2048, 2048, "pair256"), ("cta_bn256", 512, 1024, "persistent256"),
         ("cta_bn128", 384, 768, "persistent128"), ("cta_bn64", 384, 640, "persistent64"),
         ("skinny", 64, 4096, None)]


@pytest.mark.parametrize("name,M,K,cfg", DENSE, ids=[d[0] for d in DENSE])
def test_pingpong_chain(tg, monkeypatch, name, M, K, cfg):
    """X1 = X0·W, X0 = X1·W, …: each launch reads what the previous one wrote
    and overwrites what it read."""
    if cfg is None:
        monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    else:
        monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    w = _weights(K, K, 11)
    g = torch.Generator().manual_seed(12)
    x0 = torch.randn(M, K, generator=g).half()

    def make():
        return {"x0": x0.cuda(), "x1": torch.zeros(M, K, dtype=torch.half, device="cuda")}

    def step(i, b):
        src, dst = ("x0", "x1") if i % 2 == 0 else ("x1", "x0")
        tg.gemm(b[src], w, out=b[dst])

    _same(tg, step, make)


def test_mixed_kernel_chain(tg, monkeypatch):
    """Pair kernel and skinny kernel alternating on shared buffers: the
    skinny launch reads rows the pair launch just wrote, the next pair launch
    reads what the skinny one wrote into its rows."""
    monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    n = 2048
    w = _weights(n, n, 21)
    g = torch.Generator().manual_seed(22)
    x0 = torch.randn(n, n, generator=g).half()

    def make():
        return {"x0": x0.cuda(), "x1": torch.zeros(n, n, dtype=torch.half, device="cuda"),
                "y": torch.zeros(64, n, dtype=torch.half, device="cuda")}

    def step(i, b):
        if i % 4 == 0:
            tg.gemm(b["x0"], w, out=b["x1"])            # pair: X1 = X0·W
        elif i % 4 == 1:
            tg.gemm(b["x1"][:64], w, out=b["y"])        # skinny: Y = X1[:64]·W
        elif i % 4 == 2:
            tg.gemm(b["x1"], w, out=b["x0"])            # pair: X0 = X1·W
        else:
            tg.gemm(b["y"], w, out=b["x1"][:64])        # skinny: X1[:64] = Y·W

    _same(tg, step, make)


def test_sp24_chain(tg, monkeypatch):
    """2:4 sparse A fixed, B = the previous output (square, so it fits)."""
    monkeypatch.delenv("TGEMM_FORCE_SP24", raising=False)
    n = 1024
    Ac, E = W.draw_sp24(np.random.default_rng(31), n, n, ("normal", 0.0, 1.0 / np.sqrt(n / 2)))
    ac = torch.from_numpy(Ac).cuda()
    e = torch.from_numpy(E.view(np.int32)).cuda()
    g = torch.Generator().manual_seed(32)
    x0 = torch.randn(n, n, generator=g).half()

    def make():
        return {"x0": x0.cuda(), "x1": torch.zeros(n, n, dtype=torch.half, device="cuda")}

    def step(i, b):
        src, dst = ("x0", "x1") if i % 2 == 0 else ("x1", "x0")
        tg.gemm_sp24(ac, e, b[src], out=b[dst])

    _same(tg, step, make)


def test_mxfp4_chain(tg):
    """MXFP4 weight fixed (N = K), A = the previous output (the skinny
    MXFP4 kernel)."""
    M, K = 64, 2048
    Bq, S = W.draw_mxfp4(np.random.default_rng(41), K, K, 118, 120)
    bq = torch.from_numpy(Bq).cuda()
    bs = torch.from_numpy(S).cuda()
    g = torch.Generator().manual_seed(42)
    x0 = torch.randn(M, K, generator=g).half()

    def make():
        return {"x0": x0.cuda(), "x1": torch.zeros(M, K, dtype=torch.half, device="cuda")}

    def step(i, b):
        src, dst = ("x0", "x1") if i % 2 == 0 else ("x1", "x0")
        tg.gemm_mxfp4(b[src], bq, bs, K, out=b[dst])

    _same(tg, step, make)


def test_skinny_two_streams(tg, monkeypatch):
    """Skinny launches on two streams at once, each stream with its own
    inputs: every result equals the one computed alone."""
    monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    M, N, K = 64, 8192, 4096
    g = torch.Generator().manual_seed(51)
    ws = [_weights(N, K, 52 + j) for j in range(2)]
    xs = [torch.randn(M, K, generator=g).half().cuda() for _ in range(2)]
    alone = [tg.gemm(xs[j], ws[j]) for j in range(2)]
    torch.cuda.synchronize()
    tg.sync_status()
    streams = [torch.cuda.Stream() for _ in range(2)]
    outs = [[torch.empty(M, N, dtype=torch.half, device="cuda") for _ in range(6)]
            for _ in range(2)]
    torch.cuda.synchronize()
    for r in range(6):
        for j in range(2):
            with torch.cuda.stream(streams[j]):
                tg.gemm(xs[j], ws[j], out=outs[j][r], stream=streams[j])
    for j in range(2):
        tg.sync_status(streams[j])
    for j in range(2):
        for r in range(6):
            assert torch.equal(outs[j][r], alone[j]), f"stream {j}, launch {r}"
