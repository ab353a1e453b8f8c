"""The replica (N > 1) path of bench.py on the CPU: two gloo ranks agree on
the max-over-ranks step time, and every non-zero rank of the reference arm
exits without work."""
import os
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    got = d.max(1.5 + rank)                      # rank-local step times
    ref = bench.run_reference(type("A", (), {"config": "tiny", "tokens": 16, "warmup": 0,
                                              "steps": 1})(), d) if rank > 0 else "skip"
    d.done()
    q.put((rank, got, ref))


def test_two_rank_max_and_reference_rank_gate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 2000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict((r, (g, ref)) for r, g, ref in (q.get(timeout=120) for _ in procs))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == 2.5 and res[1][0] == 2.5
    assert res[1][1] is None                      # rank 1 does no reference work


def test_roofline_helpers():
    sys.path.insert(0, ROOT)
    import bench
    import moe_inputs as MI
    cfg = MI.CONFIGS["dsv3"]
    b, f = bench.alg_cost("gemm1", cfg, 4096, 256)
    assert f == 2.0 * 4096 * 8 * 7168 * 4096
    assert abs(b - (256 * 4096 * 7168 * 0.53125 + 32768 * (7168 + 4 + 4096))) < 1
    pk = dict(bench.FALLBACK)
    fr = bench.fused_roofline(cfg, 4096, 256, 1e-3, pk)
    assert fr["bound"] == "hbm" and 0 < fr["frac"] < 1


def test_reference_arm_line_matches_ours():
    """The reference arm (the oracle on the host) reports the same metric,
    unit, direction and workload configuration as the GPU arm, with its own
    cpu_baseline and an e2e entry of its own value."""
    sys.path.insert(0, ROOT)
    import bench
    import moe_inputs as MI
    args = type("A", (), {"config": "tiny", "tokens": 16, "warmup": 0, "steps": 1})()
    res = bench.run_reference(args, bench.Dist())
    cfg = MI.CONFIGS["tiny"]
    assert res["impl"] == "reference"
    assert (res["metric"], res["unit"], res["higher_is_better"]) == (bench.METRIC, bench.UNIT,
                                                                     True)
    for key, val in bench.workload_config(cfg, 16).items():
        assert res["config"][key] == val
    assert res["cpu_baseline"]["kind"] == "oracle" and res["cpu_baseline"]["value"] == res["value"]
    assert res["e2e"] == {"value": res["value"], "unit": bench.UNIT, "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}
