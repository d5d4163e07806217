"""Host logic of bench.py without a GPU: the multi-rank path (world_size 2 on gloo, CPU),
the reference arm's rank behaviour, and the workload accounting."""

from __future__ import annotations

import argparse
import contextlib
import io
import json
import os
import socket

import pytest

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    w, r, local, pg = bench.dist_setup()
    try:
        assert (w, r, local) == (world, rank, rank) and pg is not None
        assert pg.get_backend() == "gloo"
        bench.barrier(pg)
        # the slowest rank's time is the job's time
        mx = bench.max_over_ranks(pg, 1.0 + rank * 2.5)
        args = argparse.Namespace(workload="kda_b1_t256_h1_d64_f32", steps=1, warmup=1, gpus=world,
                                  impl="reference")
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            bench.run_reference(args, w, r, pg)
        bench.barrier(pg)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"max": mx, "out": buf.getvalue()}, f)
    finally:
        pg.destroy_process_group()


def test_two_ranks_on_gloo(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp

    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert all(r["max"] == 3.5 for r in res)
    # rank 0 alone runs and prints the reference line; the other rank prints nothing
    assert res[1]["out"] == ""
    line = json.loads(res[0]["out"].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    del torch


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup() == (1, 0, 0, None)
    assert bench.max_over_ranks(None, 2.0) == 2.0


def test_workload_accounting_and_dispatch():
    from types import SimpleNamespace

    from inputs import workload_inputs

    # the benchmark workload's shape (its arrays are not needed for the accounting)
    x = SimpleNamespace(dtype="bf16", T_total=16384, N=2, H_k=32, H_v=32, d_k=128, d_v=128,
                        gate="channel", h0=True, beta=True)
    # 1,540 B per (token, head) at d = 128 bf16, plus h0 and ht: 815.8 MB per launch
    assert bench.algorithmic_bytes(x) == 16384 * 32 * 1540 + 2 * 32 * 2 * 4 * 128 * 128
    assert bench.forward_kernel(x, 152) == "kda_fwd_pc_kernel"  # 64 units on 152 SMs
    assert bench.forward_kernel(x, 120) == "kda_fwd_tc_kernel"  # more than half the SMs
    y = workload_inputs("kda_b1_t256_h1_d64_f32")
    assert bench.forward_kernel(y, 152) == "kda_fwd_f32_kernel"


def test_kernel_hash_ignores_comments_and_layout_only():
    """The measured-traffic key follows the code: comments and whitespace do not change it,
    string and character literals and code do."""
    code = 'int f(int a) {\n    return a + 1;  // one\n}\n/* block\n comment */ const char *s = "x // y";\n'
    same = 'int f(int a) { return a + 1; }\n// other comment\nconst char *s = "x // y";'
    assert bench._code_only(code) == bench._code_only(same)
    assert bench._code_only(code) != bench._code_only(code.replace("a + 1", "a + 2"))
    assert bench._code_only(code) != bench._code_only(code.replace('"x // y"', '"x /* y"'))
    assert "'/'" in bench._code_only("char c = '/'; // slash")
    assert len(bench.kernel_source_hash("kda_fwd_pc_kernel")) == 16


def test_headline_traffic_is_keyed_to_the_current_kernel():
    """The headline workload's measured DRAM traffic is stored under the hash of the kernel's
    sources it was captured with; a change to those sources must come with a new capture
    (else bench.py reports the traffic as null). This fails when the two drift apart."""
    keys = [h for (w, h) in bench.MEASURED_TRAFFIC if w == "kda_b2_t8192_h32_d128_bf16"]
    assert keys, "no traffic capture for the headline workload"
    assert bench.kernel_source_hash("kda_fwd_pc_kernel") in keys


@pytest.mark.parametrize("entry", ["chunk", "recurrent", "backward"])
def test_reference_arm_times_the_entry_it_names(entry):
    """--impl reference times the oracle of the entry it is given (the token recurrence, or
    its reverse-mode gradients), on the host, with the contract's line."""
    args = argparse.Namespace(workload="kda_b1_t256_h1_d64_f32", entry=entry, steps=1, warmup=3, gpus=1)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, 1, 0, None)
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["dtype"] == "f64"
    assert ("bwd" in line["metric"]) == (entry == "backward")
    assert ("recurrent" in line["metric"]) == (entry == "recurrent")
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
