"""The named synthetic workloads (no GPU): sizes, heads, RoPE base, prompt and
generation lengths, block sizes and inner steps per block as the workload
recipe states them for the five configurations, and the ragged batch's ranges."""
import pytest

from block_wise_kv_gb300.inputs import make_config


@pytest.mark.parametrize("name,batch,d_model,heads,d_h,theta,prefix,gen,block,steps,layers", [
    ("tiny", 1, 256, 4, 64, 1e4, 64, 256, 32, 4, 1),
    ("llada_single", 1, 4096, 32, 128, 5e5, 512, 256, 32, 8, 1),
    ("stack", 16, 4096, 32, 128, 5e5, 1024, 512, 32, 16, 32),
    ("long", 4, 4096, 32, 128, 5e5, 4096, 1024, 64, 32, 1),
])
def test_uniform_workloads(name, batch, d_model, heads, d_h, theta, prefix, gen, block, steps, layers):
    c = make_config(name)
    assert (c.batch, c.d_model, c.n_heads, c.head_dim, c.rope_theta) == (batch, d_model, heads, d_h, theta)
    assert c.t_prefix == [prefix] * batch and c.gen_len == [gen] * batch and c.block == [block] * batch
    assert (c.steps_per_block, c.layers) == (steps, layers)
    for b in range(batch):
        assert c.seq_len(b) == prefix + gen
        assert c.gen_len[b] % c.block[b] == 0  # whole blocks; the suffix is all [MASK]
        k = c.block_index[b]
        assert 0 <= k < gen // block
        assert c.block_start(b) == prefix + k * block


def test_tiny_uses_token_embeddings_with_mask_id_zero():
    c = make_config("tiny")
    assert c.embedding and c.vocab == 1024 and c.mask_id == 0
    assert c.gen_len[0] // c.block[0] == 8


def test_ragged_batch():
    c = make_config("ragged")
    assert c.batch == 32 and (c.d_model, c.n_heads, c.head_dim) == (4096, 32, 128)
    assert all(128 <= t <= 4096 for t in c.t_prefix)
    assert set(c.gen_len) <= {256, 512} and set(c.block) <= {16, 32, 64}
    assert len(set(c.block)) == 3 and len(set(c.t_prefix)) > 16  # actually mixed
    for b in range(c.batch):
        assert 0 <= c.block_index[b] < c.gen_len[b] // c.block[b]
        assert c.block_start(b) == c.t_prefix[b] + c.block_index[b] * c.block[b]
    assert make_config("ragged") == c  # seeded: the same batch every time
