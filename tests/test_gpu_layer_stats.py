"""Per-layer statistics (kvevict_layer_stats): tokens kept, stored and full fp16
payload, compression ratio (page "PyramidKV ...": layer_budget,
compression_ratio, tokens_kept; page "veloxquant_mlx.quantizers.keyformer
module": keyformer_fp16_bytes, full_keyformer_fp16_bytes), checked against the
rows read_state returns as the cache fills and evicts."""
import pytest

from workloads import Workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

WL = Workload("stats", batch=2, n_layers=4, n_kv_heads=3, head_dim=64, avg_budget=40, beta=1.8,
              n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=100, rope_theta=10000.0,
              gumbel_seed=3, key_seed=91, prefill=33, decode=30)


@pytest.mark.parametrize("values", [False, True], ids=["keys", "values"])
def test_layer_stats_follow_the_cache(values):
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pre, dec = wgpu.device_inputs(WL)
    h = kvx.from_workload(WL, with_values=values)
    per_token = WL.batch * WL.n_kv_heads * WL.head_dim * 2 * (2 if values else 1)

    def check():
        p = h.next_pos
        for l in range(WL.n_layers):
            st = h.layer_stats(l)
            kept = min(p, h.layer_budget(l))
            assert st["tokens_kept"] == kept
            assert st["stored_bytes"] == per_token * kept
            assert st["full_bytes"] == per_token * p
            assert st["compression_ratio"] == (p / kept if kept else 1.0)
            assert len(h.read_state(WL.batch - 1, l, WL.n_kv_heads - 1)[3]) == kept

    check()                                   # empty
    if values:
        g = torch.Generator(device="cuda").manual_seed(1)
        h.prefill(pre, values=torch.randn(pre.shape, generator=g, device="cuda").to(torch.float16))
        check()
        h.decode(dec, values=torch.randn(dec.shape, generator=g, device="cuda").to(torch.float16))
    else:
        h.prefill(pre)
        check()
        h.decode(dec)
    check()                                   # some layers full, evicting
    assert any(h.layer_stats(l)["compression_ratio"] > 1.0 for l in range(WL.n_layers))
    with pytest.raises(kvx.KVEvictError):
        h.layer_stats(WL.n_layers)
    h.close()
