"""The seeded workload recipes: shapes, value distributions and stream independence.

Every parity test and the bench draw their inputs from these recipes, so a
recipe that silently changes shape, draws from the wrong distribution, or
reuses another tensor's random stream would weaken every comparison built on
it.  The checks here need only numpy and the generator itself.
"""
import math

import numpy as np
import pytest

from dense_packed_bit_gb300 import synth


# ---------------------------------------------------------------- stream bookkeeping

class _Recorder:
    """Stand-ins for the value generators that record (seed, draws) and return zeros.

    Generating the full-size workloads (the training set alone is 100 M values) would
    take far too long for a CPU test; the recipes' shapes and seeds are what is
    checked, so read-only zero views of the right shape and dtype suffice.
    """

    def __init__(self):
        self.calls = []       # (workload, seed, kind, draws, shape)
        self.seed_of = {}     # id(array) -> seed
        self._keep = []
        self.workload = None

    def _out(self, seed, kind, draws, shape, dtype):
        a = np.broadcast_to(np.zeros((), dtype=dtype), shape)  # right shape, no memory
        self.calls.append((self.workload, int(seed), kind, int(draws), tuple(np.shape(a))))
        self.seed_of[id(a)] = int(seed)
        self._keep.append(a)
        return a

    def install(self, monkeypatch):
        n = lambda shape: int(np.prod(shape))  # noqa: E731
        monkeypatch.setattr(synth, "normal_f32",
                            lambda s, shape, sigma=1.0: self._out(s, "normal", 2 * n(shape), shape, np.float32))
        monkeypatch.setattr(synth, "normal_f16_bits",
                            lambda s, shape, sigma=1.0: self._out(s, "normal16", 2 * n(shape), shape, np.uint16))
        monkeypatch.setattr(synth, "uniform_f32",
                            lambda s, shape, lo=-1.0, hi=1.0: self._out(s, "uniform", n(shape), shape, np.float32))
        monkeypatch.setattr(synth, "uniform_f16_bits",
                            lambda s, shape, lo, hi: self._out(s, "uniform16", n(shape), shape, np.uint16))
        monkeypatch.setattr(synth, "random_bytes",
                            lambda s, nb: self._out(s, "bytes", (nb + 7) // 8, (nb,), np.uint8))
        monkeypatch.setattr(synth, "ternary_field_bytes",
                            lambda s, nb: self._out(s, "ternary", (nb + 7) // 8, (nb,), np.uint8))


def _all_workloads(rec, replicas=(0,)):
    """Every workload recipe with the index ranges the bench and the tests use.

    Workload names carry the replica, so that a stream shared between two
    replicas counts as shared between two workloads.
    """
    out = {}

    def run(name, fn):
        rec.workload = name
        out.setdefault(name, []).append(fn())

    for r in replicas:
        sfx = f"@{r}" if r else ""
        run("gpt2_mlp_up" + sfx, lambda: synth.gpt2_mlp_up_64x768x3072(replica=r))
        run("gpt2_mlp_bias" + sfx, lambda: synth.gpt2_mlp_bias_gelu_8192x768x3072(replica=r))
        for layout in ("nn", "nt", "tn"):
            run(f"square_2048_{layout}" + sfx, lambda: synth.square_2048(layout, replica=r))
        for i in range(64):
            run("gemv2_rotation" + sfx, lambda: synth.gemv_2bit_12288x1536(i, replica=r))
            run("gemv2_t_rotation" + sfx, lambda: synth.gemv_2bit_1536x12288(i, replica=r))
            run("gemv4_rotation" + sfx, lambda: synth.gemv_4bit_12288x1536(i, replica=r))
        for layer in range(16):
            for proj in ("up", "down"):
                run("ternary_encoder" + sfx, lambda: synth.ternary_encoder_layer(layer, proj, replica=r))
        for which in ("fwd", "dA", "dB"):
            run("training_set" + sfx, lambda: synth.training_set_8192(which, replica=r))
        run("training_set_all" + sfx, lambda: synth.training_set_8192_all(replica=r))
        run("gpt2_attention" + sfx, lambda: synth.gpt2_attention_4x8x512x64(replica=r))
    return out


@pytest.fixture
def recorded(monkeypatch):
    rec = _Recorder()
    rec.install(monkeypatch)
    cases = _all_workloads(rec)
    return rec, cases


def _shared_streams(rec, ignore=()):
    by_seed = {}
    for workload, seed, kind, draws, shape in rec.calls:
        if workload in ignore:
            continue
        # the bench's one-draw form of the training set is the same workload as its per-product form
        workload = workload.replace("training_set_all", "training_set")
        assert 0 <= seed < 2 ** 32, (workload, seed)
        assert draws < 2 ** 32, (workload, seed, draws)
        by_seed.setdefault(seed, set()).add((workload, kind, draws, shape))
    return {s: v for s, v in by_seed.items() if len(v) > 1}


def test_workload_streams_are_disjoint(recorded):
    """No two tensors of any workloads share a random stream.

    Stream `s` is the counters s * 2**32 + 1 .. s * 2**32 + draws, so distinct
    seeds below 2**32 with fewer than 2**32 draws each never overlap.  A seed may
    recur only inside one workload for one and the same tensor (the shared x of a
    GEMV rotation, the training set's A and B reused by dA and dB).
    """
    rec, _ = recorded
    shared = _shared_streams(rec)
    assert not shared, f"streams drawn by more than one tensor: {shared}"


def test_training_set_all_shares_one_draw(recorded):
    """The one-draw form hands out the same A, B and dC to the three products, and they are
    the tensors the per-product form draws."""
    rec, cases = recorded
    fwd, dA, dB = cases["training_set_all"][0]
    assert dA.B is fwd.B and dB.A is fwd.A and dA.A is dB.B
    drawn = [c for c in rec.calls if c[0] == "training_set_all"]
    assert len(drawn) == 3 and len({c[1] for c in drawn}) == 3
    s = rec.seed_of
    for one, per in zip((fwd, dA, dB), cases["training_set"]):
        assert (one.name, one.transA, one.transB, one.M, one.N, one.K) == \
            (per.name, per.transA, per.transB, per.M, per.N, per.K)
        assert (s[id(one.A)], s[id(one.B)]) == (s[id(per.A)], s[id(per.B)])
    per_product = [c for c in rec.calls if c[0] == "training_set"]
    assert len(per_product) == 6                 # each product draws only the two tensors it reads


def test_replica_streams_are_disjoint(monkeypatch):
    """Eight data-parallel replicas (one per GPU of a node, weak scaling) plus the
    highest replica the seed layout holds draw no stream twice."""
    rec = _Recorder()
    rec.install(monkeypatch)
    _all_workloads(rec, replicas=tuple(range(8)) + (synth.MAX_REPLICAS - 1,))
    shared = _shared_streams(rec)
    assert not shared, f"streams drawn by more than one tensor: {shared}"


@pytest.mark.parametrize("args", [(0, 1, 0, 0), (100, 1, 0, 0), (3, 0, 0, 0), (3, 1000, 0, 0),
                                  (3, 1, -1, 0), (3, 1, 1000, 0), (3, 1, 0, -1), (3, 1, 0, synth.MAX_REPLICAS)])
def test_seed_fields_range_checked(args):
    with pytest.raises(ValueError):
        synth._seed(*args)


def test_seed_layout_largest_fits():
    assert synth._seed(99, 999, 999, synth.MAX_REPLICAS - 1) < 2 ** 32
    assert synth._seed(3, 1, 5, 0) == 3001005          # replica 0 keeps the single-GPU seeds


def test_workload_stream_count(recorded):
    """The rotations really hold 64 distinct matrices and the encoder 32 distinct layers."""
    rec, _ = recorded
    seeds = {}
    for workload, seed, kind, _, _ in rec.calls:
        seeds.setdefault((workload, kind), set()).add(seed)
    for w in ("gemv2_rotation", "gemv2_t_rotation"):
        assert len(seeds[(w, "bytes")]) == 64
        assert len(seeds[(w, "uniform16")]) == 64      # scales
        assert len(seeds[(w, "normal16")]) == 1        # one x for the whole rotation
    assert len(seeds[("gemv4_rotation", "bytes")]) == 64
    assert len(seeds[("ternary_encoder", "ternary")]) == 32
    assert len(seeds[("ternary_encoder", "normal16")]) == 32
    assert len(seeds[("training_set", "normal")]) == 3    # A, B, dC
    assert len(seeds[("gpt2_mlp_bias", "normal")]) == 3   # X, W, bias


def test_packed_workload_shapes(recorded):
    _, cases = recorded
    expect = {
        "gemv2_rotation": (12288, 1536, 384, 1, 4),
        "gemv2_t_rotation": (1536, 12288, 3072, 1, 4),
        "gemv4_rotation": (12288, 1536, 768, 1, 16),
        "ternary_encoder": (None, None, None, 222, 4),
    }
    for name, (rows, cols, rb, m, ncb) in expect.items():
        for c in cases[name]:
            if rows is not None:
                assert (c.rows, c.cols) == (rows, cols), name
                assert c.codes.shape == (rows, rb), name
            assert c.codes.dtype == np.uint8
            per_byte = 2 if ncb == 16 else 4
            assert c.codes.shape == (c.rows, -(-c.cols // per_byte))
            assert c.scales.shape == (c.rows,) and c.scales.dtype == np.uint16
            assert c.X.shape == (m, c.cols) and c.X.dtype == np.uint16
            assert c.codebook.shape == (ncb,) and c.codebook.dtype == np.float32
    tern = cases["ternary_encoder"]
    assert [(c.rows, c.cols) for c in tern[:2]] == [(3072, 768), (768, 3072)]
    assert len({c.name for c in tern}) == 32


def test_gemm_workload_layouts(recorded):
    """Stored operand shapes follow the transpose flags; dA and dB reuse the forward's tensors."""
    rec, cases = recorded
    for name, cs in cases.items():
        for c in cs:
            if not isinstance(c, synth.GemmCase):
                continue
            assert c.A.shape == ((c.K, c.M) if c.transA else (c.M, c.K)), c.name
            assert c.B.shape == ((c.N, c.K) if c.transB else (c.K, c.N)), c.name
            assert c.A.dtype == np.float32 and c.B.dtype == np.float32
    fwd, dA, dB = cases["training_set"]
    assert (fwd.transA, fwd.transB, fwd.M, fwd.N, fwd.K) == (0, 0, 8192, 8192, 2048)
    assert (dA.transA, dA.transB, dA.M, dA.N, dA.K) == (0, 1, 8192, 2048, 8192)
    assert (dB.transA, dB.transB, dB.M, dB.N, dB.K) == (1, 0, 2048, 8192, 8192)
    s = rec.seed_of
    assert s[id(dA.B)] == s[id(fwd.B)]          # dA = dC B^T with the forward's B
    assert s[id(dB.A)] == s[id(fwd.A)]          # dB = A^T dC with the forward's A
    assert s[id(dA.A)] == s[id(dB.B)]           # one dC for both
    assert s[id(dA.A)] not in (s[id(fwd.A)], s[id(fwd.B)])
    sq = [cases[f"square_2048_{l}"][0] for l in ("nn", "nt", "tn")]
    assert [(c.transA, c.transB) for c in sq] == [(0, 0), (0, 1), (1, 0)]
    mlp = cases["gpt2_mlp_up"][0]
    assert (mlp.M, mlp.N, mlp.K, mlp.transA, mlp.transB) == (64, 3072, 768, 0, 0)
    assert mlp.bias is None
    lin = cases["gpt2_mlp_bias"][0]
    assert (lin.M, lin.N, lin.K, lin.transA, lin.transB) == (8192, 3072, 768, 0, 0)
    assert lin.bias.shape == (3072,) and lin.bias.dtype == np.float32


# ---------------------------------------------------------------- real values

def _fields(codes, width):
    per = 8 // width
    mask = (1 << width) - 1
    return np.stack([(codes >> (width * f)) & mask for f in range(per)])


def _chi2_uniform_ok(counts):
    """Pearson chi-square against the uniform law, accepted below mean + 6 sd."""
    k = len(counts)
    e = counts.sum() / k
    chi2 = float(((counts - e) ** 2 / e).sum())
    return chi2 < (k - 1) + 6 * math.sqrt(2 * (k - 1)), chi2


def test_gemv2_matrix_values():
    c = synth.gemv_2bit_12288x1536(0)
    assert c.codes.shape == (12288, 384) and c.codes.dtype == np.uint8
    assert np.array_equal(c.codebook, [-2.0, -1.0, 0.0, 1.0])
    f = _fields(c.codes, 2)
    for pos in range(4):                      # every field position is uniform on 0..3
        ok, chi2 = _chi2_uniform_ok(np.bincount(f[pos].reshape(-1), minlength=4))
        assert ok, (pos, chi2)
    ok, chi2 = _chi2_uniform_ok(np.bincount(c.codes.reshape(-1), minlength=256))
    assert ok, chi2
    s = c.scales.view(np.float16).astype(np.float64)
    assert s.min() >= 0.005 - 1e-6 and s.max() < 0.05
    assert abs(s.mean() - 0.0275) < 0.001
    again = synth.gemv_2bit_12288x1536(0)
    assert synth.digest(c.codes, c.scales, c.X) == synth.digest(again.codes, again.scales, again.X)
    other = synth.gemv_2bit_12288x1536(1)
    assert not np.array_equal(other.codes, c.codes) and not np.array_equal(other.scales, c.scales)
    assert np.array_equal(other.X, c.X)      # one x for the whole rotation


def test_gemv4_matrix_values():
    c = synth.gemv_4bit_12288x1536(3)
    assert c.codes.shape == (12288, 768)
    assert np.array_equal(c.codebook, synth.CODEBOOK_NQ4)
    f = _fields(c.codes, 4)
    for pos in range(2):
        ok, chi2 = _chi2_uniform_ok(np.bincount(f[pos].reshape(-1), minlength=16))
        assert ok, (pos, chi2)


def test_transposed_gemv2_matrix_values():
    c = synth.gemv_2bit_1536x12288(5)
    assert c.codes.shape == (1536, 3072) and c.X.shape == (1, 12288)
    ok, chi2 = _chi2_uniform_ok(np.bincount(c.codes.reshape(-1), minlength=256))
    assert ok, chi2
    # the same bytes as no other rotation's matrix of the same size
    assert not np.array_equal(c.codes.reshape(-1), synth.gemv_2bit_12288x1536(5).codes.reshape(-1))


def test_ternary_layer_values():
    for proj, (rows, cols) in (("up", (3072, 768)), ("down", (768, 3072))):
        c = synth.ternary_encoder_layer(2, proj)
        assert (c.rows, c.cols) == (rows, cols)
        assert np.array_equal(c.codebook, [-1.0, 0.0, 1.0, 0.0])
        f = _fields(c.codes, 2).reshape(-1)
        cnt = np.bincount(f, minlength=4)
        n = f.size
        assert cnt[3] == 0                    # field 3 never drawn
        for v, p in ((0, 0.25), (1, 0.5), (2, 0.25)):
            sd = math.sqrt(n * p * (1 - p))
            assert abs(cnt[v] - n * p) < 6 * sd, (proj, v, cnt[v], n * p)
        # activations: N(0, 1) rounded to fp16
        x = c.X.view(np.float16).astype(np.float64).reshape(-1)
        assert np.isfinite(x).all()
        assert abs(x.mean()) < 6 / math.sqrt(x.size)
        assert abs(x.std() - 1.0) < 6 * math.sqrt(0.5 / x.size) + 1e-3
    up, down = synth.ternary_encoder_layer(2, "up"), synth.ternary_encoder_layer(3, "up")
    assert not np.array_equal(up.codes, down.codes)


def test_normal_recipe_moments():
    """Box-Muller output: mean 0, variance sigma^2, fourth moment 3 sigma^4, symmetric."""
    n = 1 << 20
    z = synth.normal_f64(11, n, 1.0)
    assert abs(z.mean()) < 6 / math.sqrt(n)
    assert abs(z.var() - 1.0) < 6 * math.sqrt(2.0 / n)
    assert abs((z ** 4).mean() - 3.0) < 6 * math.sqrt(96.0 / n)
    assert abs((z > 0).mean() - 0.5) < 6 * 0.5 / math.sqrt(n)
    # the sigma argument scales the same draws
    assert np.allclose(synth.normal_f64(11, 1000, 0.02), 0.02 * z[:1000], rtol=1e-15, atol=0)


def test_normal_chunk_boundaries():
    """Normal value i comes from draws 2i and 2i+1 of its stream, on both sides of the
    generator's internal chunk boundaries, and the fp32 / fp16 forms are the fp64 value
    rounded to nearest even."""
    ch = synth._CHUNK
    n = 2 * ch + 5
    z = synth.normal_f64(21, n, 0.5)
    for i in (0, 1, ch - 1, ch, ch + 1, 2 * ch, n - 1):
        d = synth._splitmix64(21, 2, offset=2 * i)
        u1 = (float(d[0] >> np.uint64(11)) + 1.0) * 2.0 ** -53
        u2 = float(d[1] >> np.uint64(11)) * 2.0 ** -53
        want = 0.5 * math.sqrt(-2.0 * math.log(u1)) * math.cos(2.0 * math.pi * u2)
        assert abs(z[i] - want) <= 4e-16 * 3.0, (i, z[i], want)
    assert np.array_equal(synth.normal_f32(21, (n,), 0.5), z.astype(np.float32))
    assert np.array_equal(synth.normal_f16_bits(21, (n,), 0.5), z.astype(np.float16).view(np.uint16))
    w = synth._splitmix64(8, n)
    assert np.array_equal(w[ch - 2:ch + 2], synth._splitmix64(8, 4, offset=ch - 2))
    assert synth._splitmix64(8, 0).shape == (0,) and synth.normal_f32(8, (0, 3)).shape == (0, 3)


def test_streams_are_counter_windows():
    """Stream s is a window of one counter sequence: draw i of stream s + 1 is draw
    2**32 + i of stream s, and an offset start gives the same values as the prefix."""
    a = synth._splitmix64(9, 5, offset=2 ** 32)
    b = synth._splitmix64(10, 5)
    assert np.array_equal(a, b)
    full = synth._splitmix64(4, 100)
    assert np.array_equal(synth._splitmix64(4, 40, offset=60), full[60:])
