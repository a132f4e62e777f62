"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/kvevict.h declares, computes the budget taper the
pages define, and rejects invalid configurations before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvx():
    import kv_cache_attention_02_gb300 as k
    k.lib()
    return k


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(kvevict_[a-z_]+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(kvx):
    declared = _declared()
    assert {"kvevict_create", "kvevict_prefill", "kvevict_step", "kvevict_read_state"} <= declared
    lib = ctypes.CDLL(kvx.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(kvx.SIGNATURES), "python binding covers exactly the header"


def test_budgets_match_page_and_oracle(kvx, orc):
    assert kvx.budgets(12, 512, 4, 2.0) == [1019, 927, 835, 742, 650, 558, 466, 374, 282, 189, 97, 5]
    for L, avg, ns, beta in [(1, 512, 4, 2.0), (28, 512, 4, 1.0), (32, 512, 4, 2.0), (32, 2048, 4, 1.5),
                             (16, 256, 4, 1.0), (7, 100, 0, 3.0), (9, 33, 2, 1.37), (64, 4096, 8, 1.9)]:
        assert kvx.budgets(L, avg, ns, beta) == orc.budgets(L, avg, ns, beta)


@pytest.mark.parametrize("kw,frag", [
    (dict(head_dim=96), "head_dim"),
    (dict(avg_budget=4, n_sink=4), "avg_budget"),
    (dict(tau_init=-1.0), "tau"),
    (dict(tau_end=-0.5), "tau"),
    (dict(pyramid_beta=0.5), "beta"),
    (dict(max_prefill=20000), "max_prefill"),
    (dict(layer_budgets=[10, 4]), "room to evict"),
    (dict(avg_budget=8, recent=4), "room to evict"),     # budget 8 < n_sink 4 + recent 4 + 1
    (dict(recent=-1), "recent"),
    (dict(score_mode=2), "score_mode"),
    (dict(n_layers=0), "n_layers"),
    (dict(batch=0), "batch"),
    (dict(anneal_steps=-1), "anneal"),
    (dict(rope_theta=0.0), "rope_theta"),
    (dict(avg_budget=40000), "too large"),
])
def test_invalid_config_rejected_on_host(kvx, kw, frag):
    base = dict(batch=1, n_layers=2, n_kv_heads=1, head_dim=64, n_sink=4, avg_budget=64, stream=0)
    base.update(kw)
    with pytest.raises(kvx.KVEvictError) as ei:
        kvx.KVEvict(**base)
    assert ei.value.code == kvx.ERR_INVALID_ARG
    assert frag in str(ei.value)


def test_null_arguments(kvx):
    lib = kvx.lib()
    assert lib.kvevict_create(None, None, None) == kvx.ERR_INVALID_ARG
    assert lib.kvevict_step(None, None, None, None) == kvx.ERR_INVALID_ARG
    assert lib.kvevict_read_state(None, 0, 0, 0, None, None, None, None, None, None) == kvx.ERR_INVALID_ARG
    assert lib.kvevict_destroy(None) == kvx.OK
    assert "null" in kvx.last_error()
    assert lib.kvevict_state_bytes(None, None) == kvx.ERR_INVALID_ARG
    assert lib.kvevict_save_state(None, None, 0, None) == kvx.ERR_INVALID_ARG
    assert lib.kvevict_load_state(None, None, 0, None) == kvx.ERR_INVALID_ARG
    assert lib.kvevict_layer_stats(None, 0, None, None, None, None) == kvx.ERR_INVALID_ARG
