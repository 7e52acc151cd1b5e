"""The seeded input generators: the C, numpy and torch versions agree bit for bit, and the
workloads have the stated structure."""
import math

import numpy as np
import torch

from workloads import configs, rng, torch_gen


def test_splitmix64_known_values():
    # SplitMix64 with state 0: the first outputs of the published generator
    z = rng.splitmix64(0, 0, 3)
    assert [int(x) for x in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_c_generator_matches_numpy_definition():
    for seed in range(3):
        k = rng.stream_key(seed, "k")
        sk = rng.stream_key(seed, "spike")
        np.testing.assert_array_equal(rng.normal_bf16(k, seed * 7919, 1 << 20),
                                      rng.normal_bf16_reference(k, seed * 7919, 1 << 20))
        np.testing.assert_array_equal(rng.normal_bf16(k, 3, 1 << 18, spike_key=sk, spike_prob=0.01),
                                      rng.normal_bf16_reference(k, 3, 1 << 18, spike_key=sk, spike_prob=0.01))


def test_torch_generator_matches_numpy_on_cpu():
    k = rng.stream_key(11, "k")
    a = rng.normal_bf16_reference(k, 123456, 1 << 19)
    b = torch_gen.normal_bf16(k, 123456, 1 << 19, "cpu").view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(a, b)
    wl = configs.ragged(num_seqs=4)
    kt, vt, st = torch_gen.workload_kv(wl, 0, "cpu")
    kh, vh, sh = wl.kv_all(0)
    assert np.array_equal(kt.view(torch.int16).numpy().view(np.uint16), kh)
    assert np.array_equal(vt.view(torch.int16).numpy().view(np.uint16), vh)
    assert np.array_equal(st.numpy(), sh)


def test_normal_moments_and_bf16_rounding():
    x = rng.normal(rng.stream_key(1, "m"), 0, 1 << 20)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1) < 5e-3
    b = rng.f64_to_bf16_bits(np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5]))
    # ties go to even: 1 + 2^-8 -> 1.0, 1 + 3*2^-8 -> 1 + 2^-6
    assert [hex(v) for v in b] == ["0x3f80", "0x3f80", "0x3f82", "0xc020"]


def test_config_shapes():
    t = configs.tiny()
    assert t.num_pages == 8 and list(t.context_lens) == [17] and t.pages_used() == 2
    assert sorted(t.block_tables[0, 0, :2]) != [] and (t.block_tables[0, 0, 2:] == -1).all()
    ls = configs.llama_step()
    assert ls.num_pages == 4096 and ls.num_layers == 16 and ls.pages_used() == 3712
    used = ls.block_tables[ls.block_tables >= 0]
    assert len(np.unique(used)) == used.size == 3712            # no page shared
    r = configs.ragged()
    need = sum(math.ceil(int(c) / 16) for c in r.context_lens)
    assert r.num_pages == math.ceil(1.1 * need) and r.context_lens.min() >= 1 and r.context_lens.max() <= 2048
    b = configs.bandwidth()
    assert b.num_pages == 32768 and b.num_seqs == 256 and b.algorithmic_bytes() == 1074922496
    assert ls.algorithmic_bytes() == 7619504


def test_trace_requests():
    tr = configs.trace()
    assert tr.prompt_lens.min() >= 16 and tr.prompt_lens.max() <= 512
    assert tr.new_budgets.min() >= 1 and tr.new_budgets.max() <= 512
    assert (tr.prompt_lens + tr.new_budgets - 1 <= 2048).all()
    assert sorted(tr.free_order) == list(range(tr.num_pages))
