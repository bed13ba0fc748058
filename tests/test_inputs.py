"""The seeded input generator: known answers, determinism and workload structure."""
import numpy as np

from self_referential_weight_gb300 import inputs


def test_splitmix64_known_answer():
    # SplitMix64 seeded with 0 (state advanced by the golden gamma before each
    # output): its first three outputs, as published with the generator.
    u = inputs.uniforms(np.uint64(0), 0, 3)
    got = [int(v * 2.0**53) for v in u]
    want = [0xE220A8397B1DCDAF >> 11, 0x6E789E6AA1B965F4 >> 11, 0x06C45D188009454F >> 11]
    assert got == want


def test_counter_mode_offsets_agree():
    key = inputs.stream_key(7, inputs.TAG_X)
    a = inputs.uniforms(key, 0, 100)
    b = inputs.uniforms(key, 37, 20)
    np.testing.assert_array_equal(a[37:57], b)


def test_normals_moments_and_determinism():
    key = inputs.stream_key(11, inputs.TAG_X)
    n = inputs.normals(key, 400_001)
    assert n.dtype == np.float32 and n.shape == (400_001,)
    assert abs(n.mean()) < 0.01 and abs(n.var() - 1.0) < 0.01
    np.testing.assert_array_equal(n, inputs.normals(key, 400_001))
    assert not np.array_equal(n[:100], inputs.normals(inputs.stream_key(12, inputs.TAG_X), 100))


def test_w0_scale():
    W0 = inputs.make_W0(8, 64, 4, seed=2)
    assert W0.shape == (8, 196, 64) and W0.dtype == np.float32
    assert abs(W0.std() - 1 / 8) < 0.002


def test_workload_table():
    wl = inputs.WORKLOADS
    assert (wl["mid"].B, wl["mid"].T, wl["mid"].H, wl["mid"].d, wl["mid"].m) == (64, 1024, 8, 64, 196)
    assert (wl["long"].B, wl["long"].T, wl["long"].m) == (16, 8192, 196)
    assert (wl["rl"].m, wl["rl"].n_lr, wl["rl"].softmax_input) == (97, 1, True)
    assert (wl["fewshot"].m, wl["fewshot"].T, wl["fewshot"].H * wl["fewshot"].d) == (52, 26, 256)
    assert [w.seed for w in wl.values()] == [0, 1, 2, 3, 4]


def test_fewshot_episode_structure():
    wl = inputs.workload("fewshot").with_shape(B=4)
    x = inputs.make_x(wl).reshape(4, 26, 256)
    lab = x[:, :, 251:]
    # 25 support steps with one-hot labels, five of each class; empty query label
    assert np.all(lab[:, :25].sum(-1) == 1.0)
    assert np.all(np.sort(lab[:, :25].argmax(-1), axis=1) == np.repeat(np.arange(5), 5))
    assert not lab[:, 25].any()
    # label orders differ between episodes
    assert len({tuple(lab[b, :25].argmax(-1)) for b in range(4)}) > 1


def test_two_task_means_switch_at_half():
    wl = inputs.workload("long").with_shape(B=2, T=64, H=8)
    x = inputs.make_x(wl).reshape(2, 64, 512)
    a, b = x[:, :32].mean(1), x[:, 32:].mean(1)
    # within a segment the mean is a fixed mu ~ N(0, 1); across the switch it changes
    assert np.abs(a - b).mean() > 0.8
