"""The seeded input generator shared by the oracle and the CUDA path."""
import numpy as np
import torch

import lact_inputs as li


def test_splitmix64_published_sequence():
    # First outputs of the textbook SplitMix64 seeded with 1234567 (the
    # sequence published with Vigna's reference splitmix64.c).
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    assert [int(x) for x in li.splitmix_sequence(1234567, 5)] == want


def test_counter_mode_is_the_sequence_from_the_stream_key():
    seq = li.splitmix_sequence(0, 1)  # key(seed=0, stream=0) = first draw of state 0
    key = int(seq[0])
    assert np.array_equal(li.draws(0, 0, 16), li.splitmix_sequence(key, 16))


def test_normals_and_recipe_statistics():
    z = li.normal(5, 1, (400000,))
    assert abs(float(z.mean())) < 1e-2 and abs(float(z.std()) - 1.0) < 1e-2
    q = li.unit_rows(5, 2, (1000, 64))
    np.testing.assert_allclose(np.linalg.norm(q.astype(np.float64), axis=1), 1.0, atol=1e-6)
    e = li.eta(5, 4, (100000,))
    assert e.min() > 0.0 and abs(float(e.mean()) - 0.01 * 0.8063) < 2e-4  # E[softplus(N(0,1))]=0.8063
    # the same element does not depend on how many are drawn
    np.testing.assert_array_equal(li.normal(5, 1, (10,)), z[:10])


def test_bf16_storage_is_round_to_nearest_even_of_fp32():
    f = li.normal(9, 3, (5000,))
    b = li.normal(9, 3, (5000,), bf16=True)
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(b, want)
    np.testing.assert_array_equal(li.bf16_bits_to_f32(b), torch.from_numpy(f).to(torch.bfloat16).float().numpy())


def test_workload_shapes():
    w = li.WORKLOADS[1].with_tokens(256, chunk=128)
    inp = li.make_inputs(w)
    assert inp.q.shape == (1, 2, 256, 64) and inp.k.dtype == np.float32
    assert inp.W1.shape == (2, 128, 64) and inp.W2.shape == (2, 64, 128)
    w2 = li.WORKLOADS[4].with_tokens(512, n_q=64)
    inp2 = li.make_inputs(w2)
    assert inp2.k.dtype == np.uint16 and inp2.q.shape == (1, 6, 64, 128) and w2.chunk == 512
