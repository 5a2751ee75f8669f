"""The bench's roofline numerators against the figures derived from the workload statement.

Per-expert Q2_K bytes are 84 * (2*F*H/256 + H*F/256).  A call must read the fp32 router,
x, the distinct chosen experts, the bf16 shared expert with its gate vector, and write
the fp32 out.  The prefill FLOPs count two per multiply-add of the router, three expert
matrices per (token, slot) and the shared expert.  The expected values below are written
out by hand from those definitions, not computed by the bench's helpers.
"""
import pytest

import bench
import qs_inputs as qi


@pytest.mark.parametrize("name,expect", [("tiny", 64_512), ("decode_35b_a3b", 1_032_192),
                                         ("decode_h4096", 8_257_536)])
def test_q2k_expert_bytes(name, expect):
    assert bench.expert_bytes(qi.WORKLOADS[name].shape) == expect


def test_q4k_expert_bytes():
    # 144 B per 256 weights: 144 * 3 * 512 * 2048 / 256
    assert bench.expert_bytes(qi.WORKLOADS["decode_35b_a3b"].shape, "q4k") == 1_769_472


def test_decode_35b_a3b_batch1_bytes():
    # router 256*2048*4 + x 2048*2 + 8 experts + shared (3*512*2048 + 2048)*2 + out 2048*4
    total, experts = bench.algorithmic_bytes(qi.WORKLOADS["decode_35b_a3b"].shape, 1, 8)
    assert experts == 8 * 1_032_192
    assert total == 2_097_152 + 4_096 + 8_257_536 + 6_295_552 + 8_192 == 16_662_528


def test_decode_h4096_batch1_bytes():
    # router 256*4096*4 + x 4096*2 + 8 experts + shared (3*2048*4096 + 4096)*2 + out 4096*4
    total, _ = bench.algorithmic_bytes(qi.WORKLOADS["decode_h4096"].shape, 1, 8)
    assert total == 4_194_304 + 8_192 + 66_060_288 + 50_339_840 + 16_384 == 120_619_008


def test_prefill_2048_flops():
    # router 2*2048*256*2048, routed 2*2048*8*3*512*2048, shared 2*2048*(3*512*2048 + 2048)
    flops = bench.layer_flops(qi.WORKLOADS["prefill_2048"].shape, 2048)
    assert flops == 2_147_483_648 + 103_079_215_104 + 12_893_290_496
    assert round(flops / 1e9, 1) == 118.1


def test_aggregate_throughput_counts_every_rank():
    # four replicas of 8 tokens x 100 steps over the slowest rank's 0.5 s
    assert bench.aggregate_throughput(8, 100, 4, 0.5) == 6400.0


def test_recorded_traffic_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    """roofline.traffic comes from a committed ncu summary only while the kernel sources hash to
    the value recorded beside it; an edited source (or no summary) gives None."""
    import hashlib
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    (tmp_path / "profiles").mkdir()
    digest = hashlib.sha256(b"kernel v1\n").hexdigest()[:16]
    (tmp_path / "profiles" / "fused_decode_kernel_w.md").write_text(
        f"summary\n\ntraffic_bytes_per_launch: 12345\nkernel_sources_sha256_16: {digest}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", ("k.cu",))
    assert bench.recorded_traffic("w") == 12345
    assert bench.recorded_traffic("other") is None
    src.write_text("kernel v2\n")
    assert bench.recorded_traffic("w") is None
