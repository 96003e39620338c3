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

    def backward_with_state(self, w, u, k, v, gy, state_in=None, gstate_end=None):
        """The oracle's segment backward, its unscaled sum gradients converted
        to and from the (g_num, g_den, pp) planes of the library's call."""
        sin = None if state_in is None else tuple(state_in.numpy())
        adj = None
        if gstate_end is not None:
            g = gstate_end.numpy()
            adj = (g[0] * np.exp(-g[2]), g[1] * np.exp(-g[2]))
        gw, gu, gk, gv, (ga, gb) = self.o.backward_state(w, u, k, v, gy, sin, adj)
        pp = np.full(ga.shape, -1e38) if sin is None else sin[2]
        scale = np.exp(pp)
        g_start = torch.from_numpy(np.stack([ga * scale, gb * scale, pp]))
        return (torch.from_numpy(gw), torch.from_numpy(gu), torch.from_numpy(gk), torch.from_numpy(gv), g_start)

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


def _rank_backward(rank, world, port, prefix, q):
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
    _, _, start = tsplit.forward_tsplit(w, u, ks, vs, state_in, ops=ops, want_start=True)
    gw, gu, gk, gv, g0 = tsplit.backward_tsplit(w, u, ks, vs, gs, start, ops=ops)
    q.put((rank, gw.numpy(), gu.numpy(), gk.numpy(), gv.numpy(), None if g0 is None else g0.numpy()))
    dist.destroy_process_group()


@pytest.mark.parametrize("world,prefix", [(2, 0), (3, 0), (3, 9)])
def test_ranks_backward_give_the_whole_gradients(oracle, world, prefix):
    """The ranks' backward passes, run last first and chained through the
    gradients of their start states, give the whole sequence's gk, gv and
    (all-reduced) gw, gu; with a given state before the sequence, rank 0's
    gradient of it continues the backward into the tokens that made it."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_backward, args=(r, world, port, prefix, q)) for r in range(world)]
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
