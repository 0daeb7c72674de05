"""Programmatic dependent launch with a producer in front of the finalize.

The stand-in producer (moe_finalize_rmsnorm_bench_producer) signals its
dependents at its start and writes expert_out afterwards, so the finalize
launches while expert_out is still being written; its prologue (indices,
weights, gamma, L2 prefetch of the rows) runs then, and its dependency wait
must still order every read of expert_out after the producer.  Each finalize
must therefore see exactly the rows its own producer wrote."""
import numpy as np
import pytest
import torch

import moe_finalize_residual_rmsnorm_gb300 as mfr
import workloads as W
from helpers import assert_out_close, assert_residual_close, bf16_bits, f32, oracle_on

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    mfr.build()
    mfr.load_library()


def _two_sources(wl):
    a = W.make_inputs(wl, "cuda")
    b = W.make_inputs(wl.with_(seed=wl.seed + 99), "cuda")
    return a, b["expert_out"]


@pytest.mark.parametrize("wl,kw", [(W.decode(1), {}), (W.decode(8), {}), (W.decode(64), dict(variant=mfr.VARIANT_ROWS)),
                                   (W.PREFILL.with_(T=2048), {}), (W.wide(512), {})],
                         ids=["T1_cluster", "T8_cluster", "T64_rows", "T2048_stream", "wide512_stream"])
@pytest.mark.parametrize("busy", [0, 20000])
def test_each_finalize_sees_its_producers_rows(wl, kw, busy):
    inp, other = _two_sources(wl)
    sources = [inp["expert_out"].clone(), other]
    expect = []
    for src in sources:
        d = dict(inp)
        d["expert_out"] = src
        expect.append(oracle_on(d)[:2])
    T, H, k, R = wl.T, wl.H, wl.k, wl.R
    plan = mfr.Plan(T, H, k, R, enable_pdl=True, **kw)
    expert_out = torch.zeros_like(inp["expert_out"])
    n = 12
    outs = [torch.empty((T, H), dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    routs = [torch.empty_like(inp["residual"]) for _ in range(n)]
    s = torch.cuda.current_stream()
    for i in range(n):
        mfr.bench_producer(sources[i % 2], expert_out, busy_cycles=busy, enable_pdl=True, stream=s)
        plan.run(expert_out, inp["permuted_row_of"], inp["topk_weights"], inp["residual"], routs[i], inp["gamma"],
                 inp["eps"], outs[i], s)
    torch.cuda.synchronize()
    assert plan.get_status() == 0
    for i in range(n):
        want_res, want_out = expect[i % 2]
        assert_residual_close(f32(routs[i]), want_res)
        assert_out_close(bf16_bits(outs[i]), want_out)


def test_producer_finalize_pairs_in_a_cuda_graph():
    wl = W.decode(8)
    inp, other = _two_sources(wl)
    sources = [inp["expert_out"].clone(), other]
    expect = []
    for src in sources:
        d = dict(inp)
        d["expert_out"] = src
        expect.append(oracle_on(d)[:2])
    plan = mfr.Plan(8, 4096, 8, 64, enable_pdl=True)
    expert_out = torch.zeros_like(inp["expert_out"])
    n = 10
    outs = torch.empty((n, 8, 4096), dtype=torch.bfloat16, device="cuda")
    routs = torch.empty((n, 8, 4096), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(n):
                mfr.bench_producer(sources[i % 2], expert_out, busy_cycles=5000, enable_pdl=True, stream=s)
                plan.run(expert_out, inp["permuted_row_of"], inp["topk_weights"], inp["residual"], routs[i],
                         inp["gamma"], inp["eps"], outs[i], s, validate=False)
        for _ in range(3):
            g.replay()
    s.synchronize()
    for i in range(n):
        assert_residual_close(f32(routs[i]), expect[i % 2][0])
        assert_out_close(bf16_bits(outs[i]), expect[i % 2][1])


def test_producer_rejects_bad_arguments():
    lib = mfr.load_library()
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    assert lib.moe_finalize_rmsnorm_bench_producer(x.data_ptr(), x.data_ptr(), 4, 60, 0, 1, None) == 1
    assert lib.moe_finalize_rmsnorm_bench_producer(x.data_ptr() + 2, x.data_ptr(), 4, 64, 0, 1, None) == 3
    assert lib.moe_finalize_rmsnorm_bench_producer(x.data_ptr(), x.data_ptr(), 4, 64, -1, 1, None) == 1
    torch.cuda.synchronize()
