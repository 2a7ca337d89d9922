"""The benchmark's end-to-end pipeline on the GPU: every step's pinned host
outputs hold that step's own results.  Each step gets different inputs and a
slow compute phase, so a missing wait between the copy streams and the compute
stream (a read-back before its step, an upload over inputs still in use, a step
over outputs still being read back) would show as another step's values."""
import pytest
import torch

pytestmark = pytest.mark.gpu

N_STEPS = 6
SHAPE = (1 << 20,)


def _fake_step(big):
    a, b, scratch = big

    def step(ins, outs_seq, after_o=None, before_do=None):
        q, k, v, do = ins
        o, dq, dk, dv = outs_seq
        for _ in range(8):  # a few milliseconds of work ahead of the outputs
            torch.mm(a, b, out=scratch)
        torch.add(q, k, out=o)
        if after_o is not None:
            after_o()
        for _ in range(8):
            torch.mm(a, b, out=scratch)
        if before_do is not None:
            before_do()
        torch.add(do, v, out=dq)
        torch.mul(k, 2.0, out=dk)
        torch.mul(v, 3.0, out=dv)
    return step


def _expected(i):
    q, k, v, do = (float(10 * (i + 1) + t) for t in range(4))
    return (q + k, do + v, 2.0 * k, 3.0 * v)


@pytest.mark.parametrize("one_output_set", [False, True])
def test_pipelined_steps_read_back_their_own_results(one_output_set):
    import bench
    dev = torch.device("cuda")
    pin = lambda: torch.empty(SHAPE, dtype=torch.float32, pin_memory=True)
    h_in = [[pin().fill_(10 * (i + 1) + t) for t in range(4)] for i in range(N_STEPS)]
    h_out = [[pin().fill_(-1.0) for _ in range(4)] for _ in range(N_STEPS)]
    dev_set = lambda: tuple(torch.empty(SHAPE, dtype=torch.float32, device=dev) for _ in range(4))
    sets_in = [dev_set(), dev_set()]
    outs = dev_set()
    sets_out = [outs, outs] if one_output_set else [outs, dev_set()]
    big = (torch.randn(2048, 2048, device=dev), torch.randn(2048, 2048, device=dev),
           torch.empty(2048, 2048, device=dev))
    stream = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    result_of = (lambda i: outs) if one_output_set else (lambda i: sets_out[i % 2])
    e0, e1 = bench.pipelined_steps(N_STEPS, stream, up, down, _fake_step(big), sets_in, sets_out, result_of,
                                   lambda i: h_in[i], lambda i: h_out[i], one_output_set=one_output_set)
    torch.cuda.synchronize()
    assert e0.elapsed_time(e1) > 0
    for i in range(N_STEPS):
        for got, want in zip(h_out[i], _expected(i)):
            assert float(got.min()) == want and float(got.max()) == want, (i, float(got.min()), want)
