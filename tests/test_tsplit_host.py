"""The time split of one sequence over process-group ranks
(rwkv_linear_attention_backward_b300/tsplit.py) on the CPU: gloo ranks run
its host logic (the all-gather of segment states and lengths, the choice of
the segments before each rank, the state given before the sequence) with the
float64 oracle standing in for the kernels; the outputs of all ranks, put
together, are the whole sequence's.  The kernels' side of the same steps is
tests/test_tsplit_gpu.py."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))

B, C = 2, 3
CUTS = {2: [0, 41, 70], 3: [0, 37, 42, 100]}


class OracleOps:
    """forward_with_state and state_fold computed by the oracle (float64,
    CPU tensors): the test's stand-in for the CUDA entry points."""

    def __init__(self):
        import oracle

        self.o = oracle.load()

    def forward_with_state(self, w, u, k, v, state_in=None, want_y=True):
        sin = None if state_in is None else tuple(state_in.numpy())
        y, st = self.o.forward_state(w, u, k, v, sin)
        return (torch.from_numpy(y) if want_y else None), torch.from_numpy(np.stack(st))

    def backward_with_state(self, w, u, k, v, gy, state_in=None, gstate_end=None, summary=False):
        """The oracle's segment backward, its unscaled sum gradients converted
        to and from the (g_num, g_den, pp) planes of the library's call (the
        summary pass: the start-state gradient alone)."""
        sin = None if state_in is None else tuple(state_in.numpy())
        adj = None
        if gstate_end is not None:
            g = gstate_end.numpy()
            adj = (g[0] * np.exp(-g[2]), g[1] * np.exp(-g[2]))
        gw, gu, gk, gv, (ga, gb) = self.o.backward_state(w, u, k, v, gy, sin, adj)
        pp = np.full(ga.shape, -1e38) if sin is None else sin[2]
        scale = np.exp(pp)
        g_start = torch.from_numpy(np.stack([ga * scale, gb * scale, pp]))
        if summary:
            return None, None, None, None, g_start
        return (torch.from_numpy(gw), torch.from_numpy(gu), torch.from_numpy(gk), torch.from_numpy(gv), g_start)

    def adjoint_fold(self, w, adj, lengths, gstate_end=None):
        """Start-state gradients folded last to first, in unscaled form: each
        segment's own plus the next one's decayed by e^{-n w} (the
        library's wkv_adjoint_fold), returned at the first segment's pp."""
        w = w.numpy()
        a = adj.numpy()
        X = None
        if gstate_end is not None:
            g = gstate_end.numpy()
            X = (g[0] * np.exp(-g[2]), g[1] * np.exp(-g[2]))
        for i in range(a.shape[0] - 1, -1, -1):
            own = (a[i, 0] * np.exp(-a[i, 2]), a[i, 1] * np.exp(-a[i, 2]))
            dec = np.exp(-lengths[i] * w)
            X = own if X is None else (own[0] + dec * X[0], own[1] + dec * X[1])
        pp = a[0, 2]
        return torch.from_numpy(np.stack([X[0] * np.exp(pp), X[1] * np.exp(pp), pp]))

    def state_fold(self, w, states, lengths):
        if states.shape[0] == 0:
            bc = states.shape[2:]
            return torch.stack([torch.zeros(bc, dtype=torch.float64), torch.zeros(bc, dtype=torch.float64),
                                torch.full(bc, -1e38, dtype=torch.float64)])
        return torch.from_numpy(np.stack(self.o.state_fold(w, states.numpy(), lengths)))


def _inputs(T, k_std=2.5):
    sys.path.insert(0, ROOT)
    from rwkv_linear_attention_backward_b300 import inputs

    w, u, k, v, gy = inputs.training_inputs(B, T, C, seed=77, k_std=k_std)
    return w.double(), u.double(), k.double(), v.double(), gy.double()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, prefix, q):
    for p in (ROOT, TESTS):
        sys.path.insert(0, p)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    from rwkv_linear_attention_backward_b300 import tsplit

    dist.init_process_group("gloo", rank=rank, world_size=world)
    cuts = CUTS[world]
    w, u, k, v, _ = _inputs(prefix + cuts[-1])
    ops = OracleOps()
    state_in = None
    if prefix:
        state_in = torch.from_numpy(np.stack(ops.o.state(w, k[:, :prefix], v[:, :prefix], prefix)))
    a, b = prefix + cuts[rank], prefix + cuts[rank + 1]
    y, end = tsplit.forward_tsplit(w, u, k[:, a:b].contiguous(), v[:, a:b].contiguous(), state_in, ops=ops)
    q.put((rank, y.numpy(), end.numpy()))
    dist.destroy_process_group()


@pytest.mark.parametrize("world,prefix", [(2, 0), (3, 0), (3, 9)])
def test_ranks_together_give_the_whole_sequence(oracle, world, prefix):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, prefix, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted((q.get(timeout=180) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    T = prefix + CUTS[world][-1]
    w, u, k, v, _ = _inputs(T)
    y_all = oracle.forward_direct(w, u, k, v)[:, prefix:]
    y = np.concatenate([o[1] for o in out], axis=1)
    assert y.shape == y_all.shape
    np.testing.assert_allclose(y, y_all, rtol=1e-11, atol=1e-12)
    n, d, p = oracle.state(w, k, v, T)
    end = out[-1][2]
    np.testing.assert_allclose(end[2], p, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(end[0], n, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(end[1], d, rtol=1e-11, atol=1e-13)


def _rank_backward(rank, world, port, prefix, q, with_end=False):
    for p in (ROOT, TESTS):
        sys.path.insert(0, p)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    from rwkv_linear_attention_backward_b300 import tsplit

    dist.init_process_group("gloo", rank=rank, world_size=world)
    cuts = CUTS[world]
    w, u, k, v, gy = _inputs(prefix + cuts[-1], k_std=1.0)
    ops = OracleOps()
    state_in = None
    if prefix:
        state_in = torch.from_numpy(np.stack(ops.o.state(w, k[:, :prefix], v[:, :prefix], prefix)))
    a, b = prefix + cuts[rank], prefix + cuts[rank + 1]
    ks, vs, gs = (x[:, a:b].contiguous() for x in (k, v, gy))
    _, end, start = tsplit.forward_tsplit(w, u, ks, vs, state_in, ops=ops, want_start=True)
    gend = None
    if with_end:  # a gradient on the whole sequence's end state, at the end state's pp (same on every rank)
        g = torch.Generator().manual_seed(5)
        gend = torch.stack([torch.randn(B, C, generator=g, dtype=torch.float64) * 0.3,
                            torch.randn(B, C, generator=g, dtype=torch.float64) * 0.3, torch.zeros(B, C,
                                                                                                  dtype=torch.float64)])
        last = torch.empty_like(end)
        last.copy_(end)
        dist.broadcast(last, src=world - 1)
        gend[2] = last[2]
    gw, gu, gk, gv, g0 = tsplit.backward_tsplit(w, u, ks, vs, gs, start, gend, ops=ops)
    q.put((rank, gw.numpy(), gu.numpy(), gk.numpy(), gv.numpy(), None if g0 is None else g0.numpy()))
    dist.destroy_process_group()


@pytest.mark.parametrize("world,prefix,with_end", [(2, 0, False), (3, 0, False), (3, 9, False), (3, 9, True)])
def test_ranks_backward_give_the_whole_gradients(oracle, world, prefix, with_end):
    """The ranks' backward passes, run at the same time after one exchange
    of their own start-state gradients (each folded into the earlier ranks'
    end gradients), give the whole sequence's gk, gv and (all-reduced) gw,
    gu; with a given state before the sequence, rank 0's gradient of it
    continues the backward into the tokens that made it; with a gradient on
    the sequence's end state, every gradient takes it in."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_backward, args=(r, world, port, prefix, q, with_end)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted((q.get(timeout=180) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    T = prefix + CUTS[world][-1]
    w, u, k, v, gy = _inputs(T, k_std=1.0)
    gy = gy.clone()
    gy[:, :prefix] = 0.0  # the given state's tokens are outside the split sequence
    if with_end:
        g = torch.Generator().manual_seed(5)
        ga = torch.randn(B, C, generator=g, dtype=torch.float64).numpy() * 0.3
        gb = torch.randn(B, C, generator=g, dtype=torch.float64).numpy() * 0.3
        pp_end = oracle.state(w, k, v, T)[2]
        ow, ou, ok, ov, _ = oracle.backward_state(w, u, k, v, gy, None, (ga * np.exp(-pp_end), gb * np.exp(-pp_end)))
    else:
        ow, ou, ok, ov = oracle.backward_adjoint(w, u, k, v, gy)
    gk = np.concatenate([o[3] for o in out], axis=1)
    gv = np.concatenate([o[4] for o in out], axis=1)
    np.testing.assert_allclose(gk, ok[:, prefix:], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(gv, ov[:, prefix:], rtol=1e-10, atol=1e-12)
    for o in out:
        np.testing.assert_allclose(o[2], ou, rtol=1e-10, atol=1e-12)
        if not prefix:  # with a given state, its own dependence on w lies outside the split
            np.testing.assert_allclose(o[1], ow, rtol=1e-10, atol=1e-12)
    if prefix:
        g0 = out[0][5]
        adj = (g0[0] * np.exp(-g0[2]), g0[1] * np.exp(-g0[2]))
        _, _, pk, pv, _ = oracle.backward_state(w, u, k[:, :prefix], v[:, :prefix], gy[:, :prefix], None, adj)
        np.testing.assert_allclose(pk, ok[:, :prefix], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(pv, ov[:, :prefix], rtol=1e-10, atol=1e-12)
