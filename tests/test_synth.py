"""The seeded generators: determinism, shapes and the workload statistics the
configs are calibrated to (skew of the decode routing, domain-shift rank
correlation).  CPU only."""
import numpy as np

import synth


def test_stream_is_deterministic_and_split_invariant():
    k = synth._key(0, "test", 1)
    a = synth.stream_u64(k, 10_000_000)          # spans several threaded chunks
    b = synth._u64_block(k, 0, 10_000_000)
    assert np.array_equal(a, b)
    assert np.array_equal(synth.stream_bytes(k, 17), synth.stream_bytes(k, 17))
    assert not np.array_equal(synth.stream_u64(synth._key(0, "test", 2), 8), a[:8])


def test_weight_shapes_and_scale_range():
    cfg = synth.get_config("tiny")
    w13_q, w13_s, w2_q, w2_s = synth.expert_weights(cfg, 0, 5)
    assert w13_q.shape == (2 * cfg.I, cfg.H // 2) and w13_s.shape == (2 * cfg.I, cfg.H // 32)
    assert w2_q.shape == (cfg.H, cfg.I // 2) and w2_s.shape == (cfg.H, cfg.I // 32)
    s = np.concatenate([w13_s.ravel(), w2_s.ravel()])
    assert s.min() == 123 and s.max() == 127
    nib = np.concatenate([w13_q.ravel() & 15, w13_q.ravel() >> 4])
    assert np.unique(nib).size == 16


def test_activation_bf16_rounding_and_moments():
    cfg = synth.get_config("decode1")
    x = synth.activations(cfg, 0, 0, T=64)
    f = synth.bf16_bits_to_f32(x).astype(np.float64)
    assert abs(f.mean()) < 0.02 and abs(f.std() - 1.0) < 0.02


def test_decode_skew_top25_share_near_seventy_percent():
    cfg = synth.get_config("decode1")
    lg = synth.router_logits(cfg, 0, 0, T=3000)
    ids = np.argsort(-lg, axis=1, kind="stable")[:, :cfg.k]
    cnt = np.sort(np.bincount(ids.ravel(), minlength=cfg.E))[::-1]
    share = cnt[: cfg.E // 4].sum() / cnt.sum()
    assert 0.66 <= share <= 0.74, share


def test_hot_mask_is_best_ranks():
    cfg = synth.get_config("decode1")
    m = synth.hot_mask(cfg, 0)
    r = synth.zipf_ranks(cfg, 0)
    assert m.sum() == 295 and np.all(r[m == 1] <= 295) and np.all(r[m == 0] > 295)
    d16 = synth.get_config("decode16")
    assert synth.hot_mask(d16, 1).sum() == 384 and synth.hot_mask(d16, 0).sum() == 295


def test_domain_shift_spearman():
    cfg = synth.get_config("adaptive")
    r0 = synth.zipf_ranks(cfg, 0)
    r1 = synth.shifted_ranks(cfg, 0, r0)
    assert abs(synth.spearman(r0, r1) - 0.15) <= 0.02
    a = synth.router_logits(cfg, 0, cfg.shift_at - 1, T=1)
    b = synth.router_logits(cfg, 0, cfg.shift_at, T=1)
    assert a.shape == b.shape


def test_prefill_has_no_bias():
    cfg = synth.get_config("prefill")
    assert np.all(synth.zipf_bias(cfg, synth.zipf_ranks(cfg, 0)) == 0)
