"""The shared seeded generators: deterministic, index-addressable, right distribution."""
import numpy as np
import torch

import qs_inputs as qi


def test_normal_is_index_addressable_and_deterministic():
    key = qi.make_key(3, 1003, qi.TAG_GATE, 17)
    full = qi.normal(key, 0, 1001)
    assert np.array_equal(full, qi.normal(key, 0, 1001))
    for s, n in [(0, 1), (1, 1), (5, 10), (6, 9), (999, 2), (500, 501)]:
        assert np.array_equal(qi.normal(key, s, n), full[s:s + n])


def test_normal_moments():
    z = qi.normal(qi.make_key(0, 0, 1), 0, 400000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    assert abs(np.mean(z ** 3)) < 0.02 and abs(np.mean(z ** 4) - 3) < 0.05


def test_keys_differ_per_tensor():
    a = qi.normal(qi.make_key(1, 1001, qi.TAG_GATE, 0), 0, 64)
    b = qi.normal(qi.make_key(1, 1001, qi.TAG_GATE, 1), 0, 64)
    c = qi.normal(qi.make_key(1, 1001, qi.TAG_UP, 0), 0, 64)
    assert not np.allclose(a, b) and not np.allclose(a, c)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    f = np.concatenate([rng.standard_normal(10000).astype(np.float32),
                        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)], np.float32)])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(qi.f32_to_bf16_bits(f), ref)
    assert np.array_equal(qi.bf16_bits_to_f32(ref), torch.from_numpy(f).to(torch.bfloat16).float().numpy())


def test_workload_shapes():
    w = qi.WORKLOADS
    assert w["decode_35b_a3b"].shape.expert_bytes == 1032192
    assert w["decode_h4096"].shape.expert_bytes == 8257536
    assert w["tiny"].shape.expert_bytes == 64512
    assert w["decode_35b_a3b"].copies * 256 * 1032192 == 1056964608


def test_zipf_bias_is_a_permuted_log_rank():
    sh = qi.WORKLOADS["verify8_zipf"].shape
    b = qi.gen_bias(sh, 2, 0, 1.1)
    assert np.allclose(np.sort(b)[::-1], (-1.1 * np.log(np.arange(1, 257))).astype(np.float32))
    assert qi.gen_bias(sh, 2, 0, 0.0) is None
