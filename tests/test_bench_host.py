"""Host logic of bench.py, without a GPU: byte model, L2 rotation, and the
multi-rank aggregation (world size 2 over gloo on the CPU)."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_algorithmic_bytes_per_position():
    # sliding: 8 KV heads x 256 dims x 2 bytes x (K and V) = 8192 bytes per visible position
    assert bench.algorithmic_bytes("sliding", [1], 1024) - bench.algorithmic_bytes("sliding", [0], 1024) == 8192
    # global: 1 x 512 x 2 x 2 = 2048 bytes per position
    assert bench.algorithmic_bytes("global", [10], 0) - bench.algorithmic_bytes("global", [9], 0) == 2048
    # the window caps the visible positions
    assert bench.algorithmic_bytes("sliding", [5000], 1024) == bench.algorithmic_bytes("sliding", [1024], 1024)
    # q and o: B x 16 x D x 2 bytes each (bf16 out)
    assert bench.algorithmic_bytes("global", [0, 0], 0) == 2 * 16 * 512 * 2 * 2


def test_values_only_cache_reads_half_the_bytes_per_position():
    # V only: 512 bf16 per visible position; q, o and w_k on top
    assert bench.shared_bytes([10], 0) - bench.shared_bytes([9], 0) == 1024
    assert bench.shared_bytes([5000], 100) == bench.shared_bytes([100], 100)
    assert bench.shared_bytes([0], 0) == 16 * 512 * 2 * 2 + 512 * 2


def test_append_bytes_per_token():
    # sliding: qkv row 8192 x 2 read, q 16 x 256 x 2 written, k and v 8 x 256 x 2 each written
    assert bench.append_bytes("sliding", 2) - bench.append_bytes("sliding", 1) == 16384 + 8192 + 8192
    # global: qkv row 8704 x 2 read, q 16 x 512 x 2 written, one key and one value row of 512 x 2
    assert bench.append_bytes("global", 2) - bench.append_bytes("global", 1) == 17408 + 16384 + 2048
    # the two weight vectors are read once per call
    assert bench.append_bytes("global", 0) == 2 * 512 * 2


def test_prefill_flops_count_visible_keys():
    # a 3-token prompt from scratch: queries at 0, 1, 2 see 1 + 2 + 3 keys; 4 D flops per key per head
    assert bench.prefill_flops([3], [3], 0, 8, Hq=1) == 4 * 8 * 6
    # a window of 2 caps them: 1 + 2 + 2
    assert bench.prefill_flops([3], [3], 2, 8, Hq=1) == 4 * 8 * 5
    # the last 2 tokens of 10 sit at positions 8 and 9
    assert bench.prefill_flops([10], [2], 0, 8, Hq=2) == 4 * 8 * 2 * (9 + 10)


def test_rotation_exceeds_l2():
    n = bench.rotation_count(67 * 10**6)
    assert n * 67 * 10**6 > 3 * bench.L2_BYTES
    assert bench.rotation_count(4 * 10**9) == 1


def test_aggregate_single_rank():
    line = bench.aggregate([{"bytes": 2e9, "ms": 1000.0, "calls": 10}], 10, 3, 1, {"workload": "x"})
    assert line["value"] == 2.0 and line["unit"] == "GB/s" and line["calls_per_s"] == 10.0
    assert line["ms_per_step"] == 100.0 and line["higher_is_better"] is True


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench as b
    r, w, lr = b.init_dist()
    b.setup_pg(w, "gloo")
    res = {"bytes": 1e9 * (rank + 1), "ms": 100.0 * (rank + 1), "calls": 5}
    b.barrier(w)
    allres = b.gather_results(res, w)
    if r == 0:
        q.put(b.aggregate(allres, 5, 3, w, {"workload": "x"}))
    b._PG.destroy_process_group()


def test_two_rank_aggregation_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    line = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # bytes of both ranks over the slowest rank's time: 3e9 B / 0.2 s = 15 GB/s
    assert line["value"] == 15.0
    assert line["n_gpus"] == 2 and line["scaling"] == "weak"
    assert line["calls_per_s"] == 50.0


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "0", "--config", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_recorded_traffic_tracks_the_kernel_sources():
    # a capture is reported only while the kernel sources hash to the recorded value
    for (kind, cfg), (nbytes, sha) in bench.NCU_TRAFFIC.items():
        got = bench.recorded_traffic(kind, cfg)
        assert got in (None, nbytes)
        assert (got is not None) == (bench.kernel_source_hash(kind) == sha)
    assert bench.recorded_traffic("global", "no-such-workload") is None


def test_source_hash_ignores_comments_only():
    code = "int f(int x) {\n  return x + 1;  // one more\n}\n"
    assert bench._code_only(code) == bench._code_only("/* header */\n" + code.replace("// one more", "// changed"))
    assert bench._code_only(code) != bench._code_only(code.replace("x + 1", "x + 2"))


def test_step_layers_of_one_type_share_a_page_layout():
    # The 48-layer step: each layer has its own cache and queries, and the
    # layers of one type share one page layout (one block table per type),
    # so the end-to-end loop copies each table once per step.
    from workloads import config_case, make_case
    a = config_case(5, layer=0, poison=False)
    b = config_case(5, layer=6, poison=False)
    assert a.kind == b.kind == "sliding"
    assert a.block_table.equal(b.block_table)
    assert not a.q.equal(b.q) and not a.k_pool.equal(b.k_pool)
    # the layout follows layout_seed alone; without it, the case seed
    lens = [3, 40, 100]
    c1 = make_case("global", lens, seed=1, layout_seed=9)
    c2 = make_case("global", lens, seed=2, layout_seed=9)
    c3 = make_case("global", lens, seed=9)
    assert c1.block_table.equal(c2.block_table) and c1.block_table.equal(c3.block_table)
    assert not c1.q.equal(c2.q)
    assert not make_case("global", lens, seed=1).block_table.equal(c1.block_table)
