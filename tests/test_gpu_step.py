"""Whole-step parity through the C ABI: sf_train_step against the CPU oracle
on the same seeded weights, tokens and labels.

Bar: loss relative error <= 1e-3; per-tensor gradient relative L2 error
<= 2e-2 (bf16 compute with fp32 accumulation against the float64 oracle)."""
import numpy as np
import pytest

import inputs
import oracle
from inputs import CONFIGS, TEST_CONFIGS, UNIT_EMBED, UNIT_FINAL_NORM, UNIT_LM_HEAD, IGNORE_INDEX
from inputs.configs import layer_tensor_shapes
from tests.helpers import GRAD_RL2, LOSS_RTOL, masters, oracle_weights, rel_l2

pytestmark = pytest.mark.gpu
sf = pytest.importorskip("offloaded_fine_tuning_gb300")


def make_model(cfg, mast, **kw):
    """An engine with the unit masters loaded.  Deterministic by default: the
    bitwise comparisons below need bit-reproducible attention backward sums."""
    kw.setdefault("retain_grads", 1)
    kw.setdefault("deterministic", 1)
    m = sf.Model(sf.make_config(cfg, **kw))
    for u, a in mast.items():
        m.load(u, a)
    return m


def compare(cfg, m, loss_ref, g_ref, tol=GRAD_RL2):
    errs = {"loss": abs(m.loss() - loss_ref) / abs(loss_ref)}
    for l in range(cfg.n_layers):
        flat = m.grads(l)
        off = 0
        for name, shape in layer_tensor_shapes(cfg):
            n = int(np.prod(shape))
            errs[f"{l}.{name}"] = rel_l2(flat[off:off + n].reshape(shape), g_ref["layers"][l][name])
            off += n
    errs["embed"] = rel_l2(m.grads(UNIT_EMBED).reshape(cfg.vocab, cfg.hidden), g_ref["embed"])
    errs["final_norm"] = rel_l2(m.grads(UNIT_FINAL_NORM), g_ref["final_norm"])
    if g_ref["lm_head"] is not None:
        errs["lm_head"] = rel_l2(m.grads(UNIT_LM_HEAD).reshape(cfg.vocab, cfg.hidden), g_ref["lm_head"])
    else:  # tied: no separate unit
        assert m.numel(UNIT_LM_HEAD) == 0
    bad = {k: v for k, v in errs.items() if v > (LOSS_RTOL if k == "loss" else tol)}
    assert not bad, f"outside tolerance: {bad}"
    return errs


@pytest.mark.parametrize("det", [1, 0])
@pytest.mark.parametrize("name", ["tiny", "small-gqa", "small-hd128"])
def test_step_matches_oracle(name, det):
    cfg = CONFIGS.get(name) or TEST_CONFIGS[name]
    sf.lib(build_if_needed=True)
    mast = masters(cfg)
    tok, lab = inputs.tokens_and_labels(cfg)
    loss_ref, g_ref = oracle.step(oracle_weights(cfg, mast), tok, lab, cfg)
    with make_model(cfg, mast, deterministic=det) as m:
        assert m.train_step(tok, lab) == sf.SF_OK, m.error()
        compare(cfg, m, loss_ref, g_ref)
        if det:  # a second identical step is bit-identical (no state leaks between steps)
            g0, l0 = m.grads(0), m.loss()
            assert m.train_step(tok, lab) == sf.SF_OK
            assert m.loss() == l0 and np.array_equal(m.grads(0), g0)


# ------------------------------------------------------------------ model variants
@pytest.mark.parametrize("bias,tied", [(True, True), (True, False), (False, True)])
def test_variant_step_matches_oracle(bias, tied):
    """Qwen-style Q/K/V biases and a tied LM head against the oracle."""
    cfg = TEST_CONFIGS["small-qwen"].with_(qkv_bias=bias, tie_embeddings=tied)
    mast = masters(cfg)
    tok, lab = inputs.tokens_and_labels(cfg)
    loss_ref, g_ref = oracle.step(oracle_weights(cfg, mast), tok, lab, cfg)
    with make_model(cfg, mast) as m:
        assert m.train_step(tok, lab) == sf.SF_OK, m.error()
        compare(cfg, m, loss_ref, g_ref)


def test_tied_variant_adam_tracks_oracle():
    """Two Adam steps of the biased, tied model: the embedding (also the LM
    head) and a layer's weights follow the oracle's updates."""
    cfg = TEST_CONFIGS["small-qwen"].with_(n_layers=2)
    mast = masters(cfg)
    tok, lab = inputs.tokens_and_labels(cfg)
    lr = 1e-4  # as in the multi-step test above: updates well above the bf16 noise of a step
    adam = sf.Adam(lr=lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    theta = {u: a.astype(np.float32).copy() for u, a in mast.items()}
    mom = {u: (np.zeros_like(a), np.zeros_like(a)) for u, a in theta.items()}
    for asyn in (0, 1):
        th_ = {u: a.copy() for u, a in theta.items()}
        mo_ = {u: (a.copy(), b.copy()) for u, (a, b) in mom.items()}
        with make_model(cfg, mast, async_update=asyn) as m:
            for t in range(1, 3):
                loss_ref, g = oracle.step(oracle_weights(cfg, th_), tok, lab, cfg)
                assert m.train_step(tok, lab, adam) == sf.SF_OK, m.error()
                assert abs(m.loss() - loss_ref) / loss_ref < LOSS_RTOL
                for u in th_:
                    gu = (np.concatenate([g["layers"][u][n].reshape(-1) for n, _ in layer_tensor_shapes(cfg)])
                          if u >= 0 else {UNIT_EMBED: g["embed"], UNIT_FINAL_NORM: g["final_norm"]}[u].reshape(-1))
                    th, mm, vv = oracle.adam_update(th_[u], gu.astype(np.float32), *mo_[u], t, lr)
                    th_[u], mo_[u] = th.astype(np.float32), (mm.astype(np.float32), vv.astype(np.float32))
            m.sync()
            for u in (0, UNIT_EMBED, UNIT_FINAL_NORM):
                w = m.weights(u)
                assert rel_l2(w - mast[u], th_[u] - mast[u]) < 0.1, u
                assert rel_l2(w, th_[u]) < 1e-3, u


@pytest.mark.parametrize("name,n_micro", [("small-gqa", 2), ("small-qwen", 3)])
def test_gradient_accumulation_matches_the_full_batch(name, n_micro):
    """n_micro micro-batches summed on the host equal the oracle's step on the
    whole batch (global-mean loss over every valid label)."""
    cfg = TEST_CONFIGS[name].with_(batch=n_micro)
    mast = masters(cfg)
    tok, lab = inputs.tokens_and_labels(cfg)
    lab = lab.copy()
    lab[0, :37] = IGNORE_INDEX  # micro-batches with different valid counts
    loss_ref, g_ref = oracle.step(oracle_weights(cfg, mast), tok, lab, cfg)
    micro = cfg.with_(batch=1)
    with make_model(micro, mast) as m:
        assert m.train_step_accum(tok[:, None, :], lab[:, None, :]) == sf.SF_OK, m.error()
        compare(cfg, m, loss_ref, g_ref)
        # a plain step afterwards reports its own (bf16) gradients again
        assert m.train_step(tok[:1], lab[:1]) == sf.SF_OK
        _, g1 = oracle.step(oracle_weights(cfg, mast), tok[:1], lab[:1], micro)
        assert rel_l2(m.grads(0)[:cfg.hidden], g1["layers"][0]["g1"]) < GRAD_RL2


def test_gradient_accumulation_adam_uses_the_summed_gradient():
    """An accumulated Adam step (updates overlapping the last micro-batch)
    applies Adam to the summed gradient that sf_get_grads reports, and its
    loss is the full batch's."""
    cfg = TEST_CONFIGS["small-gqa"].with_(n_layers=2, batch=2)
    mast = masters(cfg)
    tok, lab = inputs.tokens_and_labels(cfg)
    lr, wd = 1e-3, 0.01
    adam = sf.Adam(lr=lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=wd)
    with make_model(cfg, mast) as full:
        assert full.train_step(tok, lab) == sf.SF_OK
        lref = full.loss()
    with make_model(cfg.with_(batch=1), mast, async_update=1) as acc:
        assert acc.train_step_accum(tok[:, None, :], lab[:, None, :], adam) == sf.SF_OK
        assert abs(acc.loss() - lref) <= 1e-5 * lref
        acc.sync()
        for u in (0, 1, UNIT_EMBED, UNIT_LM_HEAD, UNIT_FINAL_NORM):
            g = acc.grads(u)
            z = np.zeros_like(g)
            want, _, _ = oracle.adam_update(mast[u], g, z, z, 1, lr, weight_decay=wd)
            got = acc.weights(u)
            assert rel_l2(got - mast[u], want.astype(np.float32) - mast[u]) < 1e-4, u


def test_gradient_accumulation_rejects_a_bad_micro_batch_before_running():
    cfg = TEST_CONFIGS["small-gqa"].with_(n_layers=2, batch=1)
    mast = masters(cfg)
    tok, lab = inputs.tokens_and_labels(cfg.with_(batch=3))
    tok = tok.copy()
    tok[2, 5] = cfg.vocab  # only the last micro-batch is bad
    with make_model(cfg, mast) as m:
        assert m.train_step_accum(tok[:, None, :], lab[:, None, :]) == sf.SF_EINVAL
        assert "token" in m.error()
        assert m.train_step(tok[:1], lab[:1]) == sf.SF_OK


# ------------------------------------------------------------------ optimizer state
ALL_UNITS = (0, 1, UNIT_EMBED, UNIT_LM_HEAD, UNIT_FINAL_NORM)


@pytest.mark.parametrize("tied", [False, True])
def test_bf16_adam_state_matches_oracle_elementwise(tied):
    """The host update with bf16 moments against the oracle on the same
    inputs (the engine's own gradients, weights and moments): moments bit for
    bit (same stochastic-rounding bits), weights to float32 rounding."""
    cfg = TEST_CONFIGS["small-qwen"].with_(n_layers=2, tie_embeddings=tied)
    mast = masters(cfg)
    tok, lab = inputs.tokens_and_labels(cfg)
    lr, wd = 1e-3, 0.01
    adam = sf.Adam(lr=lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=wd)
    units = [u for u in ALL_UNITS if inputs.unit_numel(cfg, u)]
    with make_model(cfg, mast, bf16_adam_state=1) as m:
        for t in (1, 2):
            before = {u: (m.weights(u), *m.adam_state(u)) for u in units}
            assert m.train_step(tok, lab, adam) == sf.SF_OK, m.error()
            assert m.adam_step == t
            for u in units:
                w0, m0, v0 = before[u]
                want, mq, vq = oracle.adam_update_bf16_states(w0, m.grads(u), m0, v0, t, lr, unit=u,
                                                              weight_decay=wd)
                m1, v1 = m.adam_state(u)
                assert np.array_equal(m1, mq) and np.array_equal(v1, vq), u
                # the engine folds the bias corrections into two constants: the
                # same update up to float32 rounding (a few ulps of the update
                # term, two of the new weight)
                w1 = m.weights(u)
                tol = 2 * np.spacing(np.abs(want)) + 5e-7 * np.abs(want - w0)
                assert np.all(np.abs(w1 - want) <= tol), u


@pytest.mark.parametrize("bf16_state", [0, 1])
def test_checkpoint_and_resume_is_bitwise(bf16_state):
    """Weights, moments and step count saved after two steps and loaded into a
    fresh engine: the third step is bit-identical to the uninterrupted run."""
    cfg = TEST_CONFIGS["small-qwen"].with_(n_layers=2)
    mast = masters(cfg)
    batches = [inputs.tokens_and_labels(cfg, seed=70 + i) for i in range(3)]
    adam = sf.Adam(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    units = [u for u in ALL_UNITS if inputs.unit_numel(cfg, u)]
    with make_model(cfg, mast, bf16_adam_state=bf16_state, async_update=1) as a:
        for tk, lb in batches[:2]:
            a.step(tk, lb, adam)
        snap = {u: (a.weights(u), *a.adam_state(u)) for u in units}
        t = a.adam_step
        loss_a = a.step(*batches[2], adam)
        after_a = {u: a.weights(u) for u in units}
    with make_model(cfg, {u: w for u, (w, _, _) in snap.items()}, bf16_adam_state=bf16_state) as b:
        for u, (_, mm, vv) in snap.items():
            b.set_adam_state(u, mm, vv)
        b.adam_step = t
        loss_b = b.step(*batches[2], adam)
        assert loss_b == loss_a
        for u in units:
            assert np.array_equal(b.weights(u), after_a[u]), u


def test_bf16_adam_state_tracks_fp32_state_training():
    """Three Adam steps with compressed moments stay with fp32 moments."""
    cfg = TEST_CONFIGS["small-gqa"].with_(n_layers=2)
    mast = masters(cfg)
    batches = [inputs.tokens_and_labels(cfg, seed=80 + i) for i in range(3)]
    adam = sf.Adam(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    out = []
    for st in (0, 1):
        with make_model(cfg, mast, bf16_adam_state=st) as m:
            losses = [m.step(tk, lb, adam) for tk, lb in batches]
            out.append((losses, {u: m.weights(u) for u in ALL_UNITS}))
    for l0, l1 in zip(out[0][0], out[1][0]):
        assert abs(l0 - l1) / l0 < 1e-4
    for u in ALL_UNITS:
        d0, d1 = out[0][1][u] - mast[u], out[1][1][u] - mast[u]
        assert rel_l2(d1, d0) < 0.05, u


# ------------------------------------------------------------------ fp16 gradients
@pytest.mark.parametrize("name", ["small-gqa", "small-qwen"])
def test_fp16_gradients_match_oracle(name):
    """Weight gradients sent as loss-scaled fp16 and unscaled on the host."""
    cfg = TEST_CONFIGS[name]
    mast = masters(cfg)
    tok, lab = inputs.tokens_and_labels(cfg)
    loss_ref, g_ref = oracle.step(oracle_weights(cfg, mast), tok, lab, cfg)
    with make_model(cfg, mast, fp16_grads=1) as m:
        assert m.train_step(tok, lab) == sf.SF_OK, m.error()
        compare(cfg, m, loss_ref, g_ref)
        assert m.stats()["loss_scale"] == 65536.0 and m.stats()["skipped_updates"] == 0


def test_fp16_gradient_overflow_skips_the_unit_and_halves_the_scale():
    """A scale of 2^24 overflows fp16: every unit whose gradient holds an
    infinity keeps its weights exactly, the others are updated, and the next
    step runs at half the scale."""
    cfg = TEST_CONFIGS["small-gqa"].with_(n_layers=2)
    mast = masters(cfg)
    tok, lab = inputs.tokens_and_labels(cfg)
    adam = sf.Adam(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    with make_model(cfg, mast, fp16_grads=1, loss_scale=2.0 ** 24) as m:
        assert m.train_step(tok, lab, adam) == sf.SF_OK, m.error()
        st = m.stats()
        assert st["loss_scale"] == 2.0 ** 24 and st["skipped_updates"] > 0
        skipped = 0
        for u in (0, 1, UNIT_LM_HEAD, UNIT_FINAL_NORM):
            if np.isfinite(m.grads(u)).all():
                assert not np.array_equal(m.weights(u), mast[u]), u
            else:
                skipped += 1
                assert np.array_equal(m.weights(u), mast[u]), u
        assert skipped == st["skipped_updates"]
        assert not np.array_equal(m.weights(UNIT_EMBED), mast[UNIT_EMBED])  # bf16 input gradient
        assert m.train_step(tok, lab, adam) == sf.SF_OK
        assert m.stats()["loss_scale"] == 2.0 ** 23


def test_fp16_gradient_adam_tracks_oracle():
    cfg = CONFIGS["tiny"]
    mast = masters(cfg)
    tok, lab = inputs.tokens_and_labels(cfg)
    lr = 1e-4
    adam = sf.Adam(lr=lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    theta = {u: a.astype(np.float32).copy() for u, a in mast.items()}
    mom = {u: (np.zeros_like(a), np.zeros_like(a)) for u, a in theta.items()}
    with make_model(cfg, mast, fp16_grads=1, async_update=1) as m:
        for t in range(1, 4):
            loss_ref, g = oracle.step(oracle_weights(cfg, theta), tok, lab, cfg)
            assert m.train_step(tok, lab, adam) == sf.SF_OK, m.error()
            assert abs(m.loss() - loss_ref) / loss_ref < LOSS_RTOL
            for u in theta:
                gu = (np.concatenate([g["layers"][u][n].reshape(-1) for n, _ in layer_tensor_shapes(cfg)])
                      if u >= 0 else {UNIT_EMBED: g["embed"], UNIT_FINAL_NORM: g["final_norm"],
                                      UNIT_LM_HEAD: g["lm_head"]}[u].reshape(-1))
                th, mm, vv = oracle.adam_update(theta[u], gu.astype(np.float32), *mom[u], t, lr)
                theta[u], mom[u] = th.astype(np.float32), (mm.astype(np.float32), vv.astype(np.float32))
        m.sync()
        assert m.stats()["skipped_updates"] == 0
        for u in ALL_UNITS:
            w = m.weights(u)
            assert rel_l2(w - mast[u], theta[u] - mast[u]) < 0.1
            assert rel_l2(w, theta[u]) < 1e-3


def test_ring_size_invariance_is_bitwise():
    cfg = TEST_CONFIGS["small-gqa"].with_(n_layers=4)
    mast = masters(cfg)
    tok, lab = inputs.tokens_and_labels(cfg)
    results = []
    for R in (2, 3, 4):
        with make_model(cfg, mast, ring_slots=R) as m:
            assert m.train_step(tok, lab) == sf.SF_OK, m.error()
            results.append((m.loss(), [m.grads(u) for u in (0, 1, 2, 3, UNIT_EMBED, UNIT_LM_HEAD)]))
    for loss, gs in results[1:]:
        assert loss == results[0][0]
        for a, b in zip(gs, results[0][1]):
            assert np.array_equal(a, b)


def test_async_update_gives_bitwise_identical_training():
    """Updates overlapping the next step (async_update) change no result."""
    cfg = TEST_CONFIGS["small-gqa"].with_(n_layers=4)
    mast = masters(cfg)
    batches = [inputs.tokens_and_labels(cfg, seed=42 + i) for i in range(3)]
    adam = sf.Adam(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    units = (0, 3, UNIT_EMBED, UNIT_LM_HEAD, UNIT_FINAL_NORM)
    out = []
    for asyn in (0, 1):
        with make_model(cfg, mast, async_update=asyn, ring_slots=2) as m:
            losses = [m.step(t, l, adam) for t, l in batches]
            m.sync()
            out.append((losses, [m.weights(u) for u in units], [m.grads(u) for u in units]))
    assert out[0][0] == out[1][0]
    for a, b in zip(out[0][1] + out[0][2], out[1][1] + out[1][2]):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("layers,asyn", [(6, 0), (6, 1), (3, 0)])
def test_sliding_activations_are_bitwise_identical(layers, asyn):
    """Checkpoints copied to the host after the forward and brought back for
    the backward (a 4-slot device window) change no result."""
    cfg = TEST_CONFIGS["small-gqa"].with_(n_layers=layers)
    mast = masters(cfg)
    batches = [inputs.tokens_and_labels(cfg, seed=50 + i) for i in range(2)]
    adam = sf.Adam(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    units = (0, layers - 1, UNIT_EMBED, UNIT_LM_HEAD)
    out, d2h = [], []
    for off in (0, 1):
        with make_model(cfg, mast, ring_slots=2, async_update=asyn, offload_activations=off) as m:
            losses = [m.step(t, l, adam) for t, l in batches]
            m.sync()
            out.append((losses, [m.grads(u) for u in units], [m.weights(u) for u in units]))
            d2h.append(m.stats()["d2h_bytes"])
    # every layer's fp32 checkpoint went to the host once per step
    assert d2h[1] - d2h[0] == layers * cfg.batch * cfg.seq * cfg.hidden * 4
    assert out[0][0] == out[1][0]
    for a, b in zip(out[0][1] + out[0][2], out[1][1] + out[1][2]):
        assert np.array_equal(a, b)


def test_lce_chunking_does_not_change_the_step():
    cfg = TEST_CONFIGS["small-gqa"]
    mast = masters(cfg)
    tok, lab = inputs.tokens_and_labels(cfg)
    out = []
    for chunk in (0, 96, 400):
        with make_model(cfg, mast, lce_chunk_rows=chunk) as m:
            assert m.train_step(tok, lab) == sf.SF_OK, m.error()
            out.append((m.loss(), m.grads(1), m.grads(UNIT_LM_HEAD)))
    for loss, g1, glm in out[1:]:
        assert abs(loss - out[0][0]) <= 1e-6 * abs(out[0][0])
        assert rel_l2(g1, out[0][1]) < 1e-3 and rel_l2(glm, out[0][2]) < 1e-3


def test_multi_step_adam_tracks_oracle():
    cfg = CONFIGS["tiny"]
    mast = masters(cfg)
    tok, lab = inputs.tokens_and_labels(cfg)
    lr = 1e-4
    adam = sf.Adam(lr=lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    # oracle: float32 masters, bf16 compute weights re-rounded after each update
    theta = {u: a.astype(np.float32).copy() for u, a in mast.items()}
    mom = {u: (np.zeros_like(a), np.zeros_like(a)) for u, a in theta.items()}
    with make_model(cfg, mast) as m:
        for t in range(1, 4):
            loss_ref, g = oracle.step(oracle_weights(cfg, theta), tok, lab, cfg)
            assert m.train_step(tok, lab, adam) == sf.SF_OK, m.error()
            assert abs(m.loss() - loss_ref) / loss_ref < LOSS_RTOL
            for u in theta:
                if u >= 0:
                    gu = np.concatenate([g["layers"][u][n].reshape(-1) for n, _ in layer_tensor_shapes(cfg)])
                else:
                    gu = {UNIT_EMBED: g["embed"], UNIT_FINAL_NORM: g["final_norm"],
                          UNIT_LM_HEAD: g["lm_head"]}[u].reshape(-1)
                th, mm, vv = oracle.adam_update(theta[u], gu.astype(np.float32), *mom[u], t, lr)
                theta[u], mom[u] = th.astype(np.float32), (mm.astype(np.float32), vv.astype(np.float32))
        for u in (0, 1, UNIT_EMBED, UNIT_LM_HEAD, UNIT_FINAL_NORM):
            w = m.weights(u)
            assert rel_l2(w - mast[u], theta[u] - mast[u]) < 0.1
            assert rel_l2(w, theta[u]) < 1e-3


def test_no_valid_label_gives_zero_loss_and_decay_only_update():
    cfg = TEST_CONFIGS["small-gqa"].with_(n_layers=2)
    mast = masters(cfg)
    tok, _ = inputs.tokens_and_labels(cfg)
    lab = np.full_like(tok, IGNORE_INDEX)
    lr, wd = 1e-2, 0.1
    with make_model(cfg, mast) as m:
        assert m.train_step(tok, lab, sf.Adam(lr=lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=wd)) == 0
        assert m.loss() == 0.0
        for u in (0, 1, UNIT_EMBED, UNIT_LM_HEAD, UNIT_FINAL_NORM):
            assert not m.grads(u).any()
            # zero gradient: Adam moves nothing but the decoupled decay
            w = m.weights(u)
            np.testing.assert_allclose(w, mast[u] * np.float32(1 - lr * wd), rtol=5e-7, atol=0)


def test_invalid_step_arguments_are_rejected():
    cfg = TEST_CONFIGS["small-gqa"].with_(n_layers=2)
    with make_model(cfg, masters(cfg)) as m:
        tok, lab = inputs.tokens_and_labels(cfg)
        bad = tok.copy(); bad[0, 3] = cfg.vocab
        assert m.train_step(bad, lab) == sf.SF_EINVAL
        badl = lab.copy(); badl[1, 0] = -5
        assert m.train_step(tok, badl) == sf.SF_EINVAL
        big = np.zeros((cfg.batch + 1, cfg.seq), dtype=np.int32)
        assert m.train_step(big, big) == sf.SF_EINVAL
        assert m.train_step(tok, lab) == sf.SF_OK  # the context is still usable


def test_adam_worker_failure_and_timeout_are_reported():
    cfg = TEST_CONFIGS["small-gqa"].with_(n_layers=2)
    tok, lab = inputs.tokens_and_labels(cfg)
    adam = sf.Adam(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    mast = masters(cfg)
    with make_model(cfg, mast, wait_timeout_ms=300) as m:
        m.inject(1, 1)          # the update of layer 1 fails on the host
        assert m.train_step(tok, lab, adam) == sf.SF_ESTATE
        assert "injected" in m.error()
        m.inject(0)
        # the failed unit kept its weights; the step after it runs normally
        np.testing.assert_array_equal(m.weights(1), mast[1])
        assert m.train_step(tok, lab, adam) == sf.SF_OK
        m.inject(2, 1500)       # host updates slower than the wait bound
        assert m.train_step(tok, lab, adam) == sf.SF_ETIMEOUT
        assert "timed out" in m.error()
        m.inject(0)


# ------------------------------------------------------------------ full-size shapes
@pytest.mark.parametrize("name,seq", [("8b", 2048), ("123b-slice", 1024)])
def test_one_full_shape_layer_matches_oracle(name, seq):
    """One decoder layer at the full width of the 8B and 123B-slice shapes
    (GQA 4:1 and 12:1, head_dim 128, full vocabulary), one sequence, against
    the float32 oracle (float32 is within ~1e-6 of float64, far inside the bar)."""
    cfg = CONFIGS[name].with_(n_layers=1, batch=1, seq=seq)
    mast = masters(cfg)
    tok, lab = inputs.tokens_and_labels(cfg)
    loss_ref, g_ref = oracle.step(oracle_weights(cfg, mast), tok, lab, cfg, dtype=np.float32)
    with make_model(cfg, mast, ring_slots=2) as m:
        assert m.train_step(tok, lab) == sf.SF_OK, m.error()
        compare(cfg, m, loss_ref, g_ref)


def test_full_1p3b_step_properties():
    """The whole 24-layer 1.3B-shape step (8 x 1024 tokens): loss near
    ln V + sigma^2/2 (random init), finite gradients, and ring sizes 2 and 3
    give bit-identical results."""
    import math
    cfg = CONFIGS["1.3b"]
    mast = masters(cfg)
    tok, lab = inputs.tokens_and_labels(cfg)
    out = []
    for R in (2, 3):
        with make_model(cfg, mast, ring_slots=R) as m:
            assert m.train_step(tok, lab) == sf.SF_OK, m.error()
            out.append((m.loss(), m.grads(0), m.grads(cfg.n_layers - 1), m.grads(UNIT_LM_HEAD)))
    loss = out[0][0]
    assert loss == pytest.approx(math.log(cfg.vocab) + 0.02 ** 2 * cfg.hidden / 2, rel=0.02)
    assert out[1][0] == loss
    for a, b in zip(out[0][1:], out[1][1:]):
        assert np.isfinite(a).all() and np.array_equal(a, b)


def depth_tolerance(name, batch):
    """Per-tensor bounds of a whole-stack comparison at the workload's depth:
    the stated bar (2e-2), or, where the bf16-operand rounding model (written
    by tests/golden/make_bf16_depth_error.py from the oracle alone) already
    moves the gradients by more, 1.25x that model's error.  The model rounds
    only where any bf16 tensor-core path must (projection and attention
    operands, P and dS, the gradient cast), so no storage choice of this path
    sets the bound.  1.25 covers the scatter between two independent
    realisations of the same rounding noise (this path's and the model's).
    Where the test runs the golden's own tokens (batch and sequence length
    equal), each tensor is also held to 1.15x the model's error for that
    very tensor."""
    import json
    import os
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                       f"bf16_depth_error_{name}.json")))
    assert gold["workload"] == CONFIGS[name].name
    k = 1.25
    return gold, {"layers": max(GRAD_RL2, k * gold["layer_max"]),
                  "median": max(GRAD_RL2, k * gold["layer_median"]),
                  "lm_head": max(GRAD_RL2, k * gold["lm_head"]),
                  "final_norm": max(GRAD_RL2, k * gold["final_norm"]),
                  "embed": max(GRAD_RL2, k * gold["embed"]),
                  # where the test runs the golden's own tokens (one sequence),
                  # each tensor against the model's error for that tensor
                  "per_tensor": ({t: max(GRAD_RL2, PER_TENSOR_K * e) for t, e in gold["per_tensor"].items()}
                                 if gold["batch"] == batch and gold["seq"] == CONFIGS[name].seq else None)}


# Per-tensor bound on the golden's own tokens: this path's error and the
# model's are two draws of the same rounding noise on the same inputs; they
# agree to a few percent of each other (medians to 0.2%), so 1.15x.
PER_TENSOR_K = 1.15


def load_streamed(cfg, m):
    """Load every unit's fp32 masters, generating one layer at a time."""
    for l in range(cfg.n_layers):
        m.load(l, inputs.layer_master(cfg, l))
    for u in (UNIT_EMBED, UNIT_FINAL_NORM, UNIT_LM_HEAD):
        m.load(u, inputs.unit_master(cfg, u))


def compare_streamed(cfg, m, tol):
    """The float32 oracle's step, layer by layer (each layer's bf16 weights
    regenerated from the seeded generator), against the engine's retained
    gradients, tensor by tensor as the oracle's backward produces them."""
    shapes = layer_tensor_shapes(cfg)
    errs = {}

    def layer(i):  # rounded tensor by tensor: smaller temporaries than the whole layer
        return {k: oracle.bf16_round(v) for k, v in inputs.split_layer(cfg, inputs.layer_master(cfg, i)).items()}

    def check(i, g):
        flat = m.grads(i)
        off = 0
        for name, shape in shapes:
            n = int(np.prod(shape))
            errs[f"{i}.{name}"] = rel_l2(flat[off:off + n].reshape(shape), g[name])
            off += n

    d, V = cfg.hidden, cfg.vocab
    r = lambda u: oracle.bf16_round(inputs.unit_master(cfg, u))
    tok, lab = inputs.tokens_and_labels(cfg)
    loss_ref, g = oracle.step_streamed(layer, cfg.n_layers, r(UNIT_EMBED).reshape(V, d),
                                       r(UNIT_FINAL_NORM), r(UNIT_LM_HEAD).reshape(V, d), tok, lab,
                                       cfg, dtype=np.float32, on_layer_grads=check)
    layer_errs = np.array(list(errs.values()))
    errs["loss"] = abs(m.loss() - loss_ref) / abs(loss_ref)
    errs["embed"] = rel_l2(m.grads(UNIT_EMBED).reshape(V, d), g["embed"])
    errs["final_norm"] = rel_l2(m.grads(UNIT_FINAL_NORM), g["final_norm"])
    errs["lm_head"] = rel_l2(m.grads(UNIT_LM_HEAD).reshape(V, d), g["lm_head"])
    errs["layer_median"] = float(np.median(layer_errs))
    errs["layer_max"] = float(layer_errs.max())
    bad = {k: v for k, v in errs.items() if k[0].isdigit() and v > tol["layers"]}
    assert not bad, f"outside tolerance {tol['layers']:.4f}: {bad}"
    if tol.get("per_tensor") is not None:
        over = {t: (v, tol["per_tensor"][t]) for t, v in errs.items()
                if t in tol["per_tensor"] and v > tol["per_tensor"][t]}
        assert not over, f"above {PER_TENSOR_K}x the model's own error for the tensor: {over}"
        ratio = [v / e for t, v in errs.items() if t in tol["per_tensor"]
                 for e in [tol["per_tensor"][t] / PER_TENSOR_K] if e > 0]
        errs["ratio_to_model_max"] = float(max(ratio))
    assert errs["loss"] <= LOSS_RTOL, errs["loss"]
    for k in ("embed", "final_norm", "lm_head"):
        assert errs[k] <= tol[k], (k, errs[k], tol[k])
    assert errs["layer_median"] <= tol["median"], (errs["layer_median"], tol["median"])
    return errs


def test_full_1p3b_step_matches_oracle():
    """The whole 1.3B-shape step (24 layers, hidden 2048, 16 x 64 heads, FFN
    5504, vocab 32000, 8 x 1024 tokens) against the float32 oracle, tensor by
    tensor (the oracle needs a couple of minutes of the host's cores).  Loss
    within 1e-3; gradients within depth_tolerance("1.3b")."""
    cfg = CONFIGS["1.3b"]
    gold, tol = depth_tolerance("1.3b", cfg.batch)
    with make_model(cfg, {}) as m:
        load_streamed(cfg, m)
        assert m.train_step(*inputs.tokens_and_labels(cfg)) == sf.SF_OK, m.error()
        errs = compare_streamed(cfg, m, tol)
    print({k: v for k, v in errs.items() if not k[0].isdigit()}, "model:", gold["layer_max"])


def test_full_8b_stack_matches_oracle():
    """The whole 32-layer 8B-shape GQA stack (hidden 4096, 32/8 heads x 128,
    FFN 14336, vocab 128256, RoPE base 500000) streamed through the 3-slot
    ring, one sequence of 2048 tokens, against the float32 oracle tensor by
    tensor.  The optimizer state is kept as bf16 (no update runs here) so the
    engine's host memory and the oracle's activations fit the host together."""
    cfg = CONFIGS["8b"].with_(batch=1)
    gold, tol = depth_tolerance("8b", cfg.batch)
    with make_model(cfg, {}, ring_slots=3, bf16_adam_state=1) as m:
        load_streamed(cfg, m)
        assert m.train_step(*inputs.tokens_and_labels(cfg)) == sf.SF_OK, m.error()
        errs = compare_streamed(cfg, m, tol)
    print({k: v for k, v in errs.items() if not k[0].isdigit()}, "model:", gold["layer_max"])


def test_full_123b_slice_matches_oracle():
    """The 123B-shape slice as configured (4 layers of hidden 12288, 96/8
    heads x 128, FFN 28672, vocab 32768, 2-slot ring), one sequence of 1024
    tokens, against the float32 oracle tensor by tensor."""
    cfg = CONFIGS["123b-slice"].with_(batch=1)
    gold, tol = depth_tolerance("123b-slice", cfg.batch)
    with make_model(cfg, {}, ring_slots=2, bf16_adam_state=1) as m:
        load_streamed(cfg, m)
        assert m.train_step(*inputs.tokens_and_labels(cfg)) == sf.SF_OK, m.error()
        errs = compare_streamed(cfg, m, tol)
    print({k: v for k, v in errs.items() if not k[0].isdigit()}, "model:", gold["layer_max"])


@pytest.mark.parametrize("asyn", [0, 1])
def test_sliding_activations_match_oracle(asyn):
    """Sliding activations (checkpoints to pinned host memory after the
    forward, back before the backward) against the oracle, tensor by tensor,
    with more layers than the 4-slot device window."""
    cfg = TEST_CONFIGS["small-gqa"].with_(n_layers=6)
    mast = masters(cfg)
    tok, lab = inputs.tokens_and_labels(cfg)
    loss_ref, g_ref = oracle.step(oracle_weights(cfg, mast), tok, lab, cfg)
    with make_model(cfg, mast, offload_activations=1, ring_slots=2, async_update=asyn) as m:
        assert m.train_step(tok, lab) == sf.SF_OK, m.error()
        compare(cfg, m, loss_ref, g_ref)
        assert m.stats()["d2h_bytes"] > cfg.n_layers * cfg.batch * cfg.seq * cfg.hidden * 4
