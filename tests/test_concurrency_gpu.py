"""Plans are independent: concurrent use of two plans gives the serial bits.

A plan owns its workspace (stream-K partial tiles and arrival counters) and its
staging buffer, and the library documents one plan per stream.  Every kernel
here reduces in a fixed order, so a result computed while another plan works on
another stream, or from another host thread, must equal the result computed
alone, bit for bit.  The shapes are chosen to use the plan's memory: the
swap-AB kernel with split tiles (partials and counters), the pair kernel's
stream-K phase (partials), and a misaligned operand (the staging copy).
"""
import threading

import pytest
import torch

import dense_gemm_05_gb300 as g

pytestmark = pytest.mark.gpu

# (M, K, N, dtype, lda pad, ldb pad)
SHAPES = [
    (16, 4096, 4864, torch.bfloat16, 0, 0),      # swap-AB stream-K, split tiles
    (4096, 4096, 4096, torch.bfloat16, 0, 0),    # pair tiles with a stream-K phase
    (1023, 640, 1029, torch.float16, 0, 0),      # B staged (ldb = 1029 halves; 10 K blocks)
    (600, 1000, 1104, torch.float16, 3, 0),      # A staged (lda = 1003 halves)
]


@pytest.fixture(scope="module")
def plans():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.build()
    ps = [g.Plan(0), g.Plan(0)]
    yield ps
    for p in ps:
        p.close()


def make(shape, seed):
    M, K, N, dt, pa, pb = shape
    dev = torch.device("cuda:0")
    gen = torch.Generator(device=dev).manual_seed(seed)
    a = torch.randn(M, K + pa, generator=gen, device=dev).to(dt)[:, :K]
    b = torch.randn(K, N + pb, generator=gen, device=dev).to(dt)[:, :N]
    return a, b


def serial(plan, a, b):
    c = torch.empty(a.shape[0], b.shape[1], dtype=torch.float32, device=a.device)
    plan.run(a, b, c)
    torch.cuda.synchronize()
    return c


def test_shapes_use_the_plan_memory(plans):
    cfgs = []
    for shape in SHAPES:
        a, b = make(shape, 1)
        c = torch.empty(a.shape[0], b.shape[1], dtype=torch.float32, device=a.device)
        cfgs.append(plans[0].query(a, b, c))
    assert cfgs[0]["kernel"] == g.GEMM_KERNEL_SKINNY and cfgs[0]["split_k"] > 1, cfgs[0]
    assert cfgs[1]["kernel"] == g.GEMM_KERNEL_PAIR and cfgs[1]["shares"] > 0, cfgs[1]
    assert cfgs[2]["staged"] & 2 and cfgs[3]["staged"] & 1, (cfgs[2], cfgs[3])


def test_two_plans_on_two_streams(plans):
    inputs = [[make(s, 10 + 2 * i + j) for j in range(2)] for i, s in enumerate(SHAPES)]
    ref = [[serial(plans[j], *inputs[i][j]) for j in range(2)] for i in range(len(SHAPES))]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[torch.full_like(ref[i][j], float("nan")) for j in range(2)]
            for i in range(len(SHAPES))]
    torch.cuda.synchronize()
    for rep in range(5):
        for i in range(len(SHAPES)):
            for j in range(2):
                plans[j].run(*inputs[i][j], outs[i][j], stream=streams[j])
        for j in range(2):
            streams[j].synchronize()
        for i in range(len(SHAPES)):
            for j in range(2):
                assert torch.equal(outs[i][j], ref[i][j]), (rep, SHAPES[i][:3], j)
                outs[i][j].fill_(float("nan"))
        torch.cuda.synchronize()


def test_two_host_threads(plans):
    inputs = [[make(s, 30 + 2 * i + j) for j in range(2)] for i, s in enumerate(SHAPES)]
    ref = [[serial(plans[j], *inputs[i][j]) for j in range(2)] for i in range(len(SHAPES))]
    errors = []

    def worker(j):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for rep in range(5):
                    for i in range(len(SHAPES)):
                        out = torch.full_like(ref[i][j], float("nan"))
                        plans[j].run(*inputs[i][j], out, stream=s)
                        s.synchronize()
                        if not torch.equal(out, ref[i][j]):
                            errors.append((j, rep, SHAPES[i][:3]))
        except Exception as e:   # surfaced below
            errors.append((j, repr(e)))

    threads = [threading.Thread(target=worker, args=(j,)) for j in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
