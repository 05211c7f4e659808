"""Host-side pieces of bench.py that need no GPU: the replicas' max-over-ranks
reduction (two gloo ranks on CPU) and the source-matched DRAM traffic record."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _fake_res(step_ms, dec_ms):
    """A pass result as run_ours returns it, for a small CPU workload."""
    from paged_kv_decode_19_gb300 import workloads as W
    wl = W.make("llama3_8b_bf16", seed=3, reduced=True, device="cpu", B=2,
                len_dist=("uniform", 5, 20))
    return dict(step=step_ms, dec=dec_ms, dec_med=dec_ms, app=0.005, dec_flushed=dec_ms,
                dec_devplan=dec_ms,
                e2e=2 * step_ms, launches=40, variant="mma", clocks=None, wl=wl, h2d=10,
                d2h=20, alternate=True, l2=1 << 27, ext=None)


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        # each replica reports its own time; every rank learns the slowest
        mx = bench._max_over_ranks(10.0 + 5.0 * rank, ws)
        # replicas: the per-call times are the slowest rank's, not divided by the ranks
        res = _fake_res(0.060 + 0.004 * rank, 0.050 + 0.004 * rank)
        # rank 1 has no graph-replayed time (its capture refused): no rank may hang on it
        res["e2e_graph"] = 0.070 if rank == 0 else None
        res["dec_b2b"] = 0.045 + 0.002 * rank
        summ = bench._summarise(res, "llama3_8b_bf16", res["wl"].spec, ws)
        q.put((rank, mx, bench._dist(), summ["step_us"], summ["decode_us"], summ["e2e"]["value"],
               summ["e2e"]["graph_replayed"], summ["decode_us_back_to_back"]))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [15.0, 15.0]
    assert [g[2][:2] for g in got] == [(2, 0), (2, 1)]  # (world size, rank) from the env
    for g in got:
        assert g[3] == 64.0 and g[4] == 54.0 and g[5] == 128.0
        assert g[6] == 70.0 and g[7] == 47.0


def test_single_rank_is_identity():
    assert bench._max_over_ranks(3.5, 1) == 3.5


def test_summary_of_one_pass():
    """Per-call times in microseconds from the pass's milliseconds; the roofline divides
    the algorithmic bytes (attended K + V, Q, out, lse) by the decode time."""
    res = _fake_res(0.060, 0.050)
    s = bench._summarise(res, "llama3_8b_bf16", res["wl"].spec, 1)
    assert s["step_us"] == 60.0 and s["decode_us"] == 50.0 and s["e2e"]["value"] == 120.0
    alg = res["wl"].kv_bytes_attended() + res["wl"].io_bytes()
    assert s["roofline"]["algorithmic_bytes"] == alg
    assert abs(s["roofline"]["achieved"] - alg / 50e-6 / 1e9) < 0.1
    assert "multi_stage" not in s and s["l2"].startswith("inputs larger than L2")


def test_traffic_record_only_for_matching_sources(tmp_path, monkeypatch):
    digest = bench._sources_digest()
    assert digest == bench._sources_digest() and len(digest) == 64
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"cfgA:B=4": {"sources_sha256": digest, "dram_bytes_per_launch": 1234},
           "cfgB:B=4": {"sources_sha256": "0" * 64, "dram_bytes_per_launch": 99}}
    (prof / "dram_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "_sources_digest", lambda: digest)
    assert bench._measured_traffic("cfgA", 4) == 1234
    assert bench._measured_traffic("cfgB", 4) is None   # taken on other sources
    assert bench._measured_traffic("cfgA", 8) is None   # another batch size


def test_append_inputs_cover_the_last_q_len_rows():
    """The step's append writes each sequence's last q_len rows (its new tokens): the
    slot of row r is page_table[r // P] * P + r % P; a row before the sequence start
    is skipped (-1)."""
    import numpy as np
    from paged_kv_decode_19_gb300 import workloads as W
    for q_len in (1, 2, 3):
        wl = W.make("llama3_8b_bf16", seed=5, reduced=True, device="cpu", q_len=q_len,
                    len_dist=("uniform", 1, 40), B=6)
        k, v, slots = bench._append_inputs(wl, "cpu")
        s = wl.spec
        assert k.shape == (s.B * q_len, s.H_kv, s.D) and v.shape == k.shape
        ip, vals, P = wl.indptr.numpy(), wl.values.numpy(), s.page_size
        got = slots.numpy().reshape(s.B, q_len)
        for b in range(s.B):
            for j in range(q_len):
                r = int(wl.seq_len[b]) - q_len + j
                want = -1 if r < 0 else int(vals[ip[b] + r // P]) * P + r % P
                assert got[b, j] == want, (q_len, b, j)


def test_spec_decode_workload_shapes_and_positions():
    from paged_kv_decode_19_gb300 import workloads as W
    wl = W.make("spec_decode_bf16", seed=6, reduced=True, device="cpu")
    s = wl.spec
    assert s.q_len == 2 and wl.Q.shape == (s.B, 2, s.H_qo, s.D)
    # token t of a sequence sits at its own row's position: L - q_len + t
    assert (wl.q_rope_position.numpy() == (wl.attended - 2).clip(min=0)).all()
    assert wl.io_bytes() == 2 * W.make("llama3_8b_bf16", seed=6, reduced=True, device="cpu").io_bytes()


def test_oracle_samples_single_and_threaded_cover_whole_sequences():
    """Both CPU-baseline samples decode whole sequences: with an ample budget every
    sequence is done exactly once and the attended rows add up; with no budget the
    single-thread sample stops after one sequence and the threaded one after its first
    wave (one sequence per thread)."""
    from paged_kv_decode_19_gb300 import workloads as W
    wl = W.make("llama3_8b_bf16", seed=7, reduced=True, device="cpu", B=5,
                len_dist=("uniform", 1, 60))
    total = int(wl.attended.sum())
    _, n1, r1 = bench._oracle_sample(wl, 1e9)
    _, n3, r3 = bench._oracle_sample_threads(wl, 1e9, 3)
    assert (n1, r1) == (5, total) and (n3, r3) == (5, total)
    _, n1, r1 = bench._oracle_sample(wl, 0.0)
    assert (n1, r1) == (1, int(wl.attended[0]))
    _, n3, r3 = bench._oracle_sample_threads(wl, 0.0, 3)
    assert (n3, r3) == (3, int(wl.attended[:3].sum()))  # the first wave, nothing after it
    line = bench._cpu_baseline(wl, 1e9)
    assert line["kind"] == "oracle" and line["cores"] == 1 and line["value"] > 0
    if bench._host_cores() > 1:
        assert line["all_cores"]["cores"] == bench._host_cores()
        assert line["all_cores"]["value"] > 0


def test_padded_chunk_split_layout():
    """Chunk j of sequence b sits at j * B + b; the chunks of a sequence hold its page
    list once, in order, and their rows add up to its length; a chunk past the end of
    the list has no pages."""
    import numpy as np
    from paged_kv_decode_19_gb300 import workloads as W
    wl = W.make("long_ctx_bf16", seed=2, reduced=True, device="cpu")
    ip, vals, B = wl.indptr.numpy(), wl.values.numpy(), wl.spec.B
    for nsplit in (1, 4, 32):
        ipc, valc, lastc, roff = W.split_chunks_padded(ip, vals, wl.seq_len, 16, nsplit)
        assert len(ipc) == nsplit * B + 1 and len(lastc) == len(roff) == nsplit * B
        for b in range(B):
            sel = [j * B + b for j in range(nsplit)]
            got = np.concatenate([valc[ipc[i]:ipc[i + 1]] for i in sel])
            assert np.array_equal(got, vals[ip[b]:ip[b + 1]])
            rows, start = 0, 0
            for i in sel:
                n = ipc[i + 1] - ipc[i]
                if n == 0:
                    continue
                assert roff[i] == start and 1 <= lastc[i] <= 16
                start += n * 16
                rows += (n - 1) * 16 + lastc[i]
            assert rows == wl.seq_len[b]


def test_multi_stage_flow_equals_unsplit_decode_in_the_oracle():
    """The bench's multi-stage flow, run with the oracle on both stages (chunk decode of
    the padded pseudo-sequences with RoPE offsets, then the halving merge tree), equals
    the oracle's unsplit decode: the re-indexing and the tree drop or repeat no row."""
    import numpy as np
    import oracle
    from paged_kv_decode_19_gb300 import workloads as W
    wl = W.make("llama3_8b_bf16", seed=8, reduced=True, device="cpu", B=3,
                len_dist=("uniform", 1, 150))
    s, nsplit = wl.spec, 8
    x = bench._external_split(wl, nsplit, "cpu")
    kw = dict(q_dtype=s.q_dtype, kv_dtype=s.kv_dtype, H_kv=s.H_kv, page_size=s.page_size,
              rotary_mode=s.rotary_mode, rope_scale=s.rope_scale, rope_theta=s.rope_theta,
              sm_scale=wl.sm_scale)
    out, lse, st = oracle.batch_decode_paged_kv(
        W.bits(x["Q"]), W.bits(wl.pages), x["indptr"].numpy(), x["values"].numpy(),
        x["length_info"].numpy(), x["k_rope_pos_offset"].numpy(),
        x["q_rope_position"].numpy(), **kw)
    assert st == 0

    def merge(V, S, Vo, So):
        V[...], S[...] = oracle.merge_state(V, S, Vo, So)

    got_o, got_l = bench._merge_tree(out, lse, nsplit, s.B, merge)
    ro, rl, st = oracle.batch_decode_paged_kv(
        W.bits(wl.Q), W.bits(wl.pages), wl.indptr.numpy(), wl.values.numpy(),
        wl.length_info.numpy(), wl.k_rope_pos_offset.numpy(), wl.q_rope_position.numpy(), **kw)
    assert st == 0
    np.testing.assert_allclose(got_o, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got_l, rl, rtol=0, atol=1e-12)


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` needs no GPU: it times the fp64 oracle and prints one
    JSON line with the arm's metric, unit and config, marked as the reference."""
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl",
                        "reference", "--config", "tiny_fp32", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=bench.ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is False and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["config"]["workload"].startswith("tiny_fp32:")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["value_is_scaled"] is True
    assert d["scaling_of_value"]["rows_per_call"] > d["scaling_of_value"]["rows_timed_per_step"] > 0
