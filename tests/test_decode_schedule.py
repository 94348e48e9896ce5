"""Host model of the Relation Cache decode's chunk schedule (no GPU).

The bulk-copy decode kernel (one cluster of S CTAs per head) streams the t cached
rows of a head in chunks of ch rows through a ring of three shared-memory stages.
CTA s of the cluster takes chunks k0 .. k0 + nck - 1 with per = ceil(n / S) chunks
per CTA, n = ceil(t / ch).  Before the position t is known, stage 0 is already
filled with a guess: the first chunk the CTA would take were the cache full
(t = T - 1), copying the allocation's rows only.  Once t is known:

- a right guess (the CTA's first chunk is the guessed one) is scored as that chunk;
- a wrong guess is consumed as an empty stage, and every later fill is shifted by
  one (lag 1).

Fill f goes to stage f mod 3 only after fill f - 3 has been consumed.  A fill with
no chunk left completes its stage's barrier without a copy and ends the loop.

For every cache size, chunk size, cluster size and position in the ranges below,
the model checks that:

- each CTA scores exactly its own chunks, in order, and stops;
- the CTAs of a cluster together cover the rows 0 .. t-1 once;
- every scored row was copied (a right guess copies at least the rows scored);
- each consumption sees the fill whose barrier phase it waits on.

Two planted mistakes must be caught: accepting any guess, and forgetting the lag.
A source check ties the modelled expressions to the kernel.
"""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "relation_token_mixing_gb300", "csrc")
STAGES = 3
EMPTY = -2


def _cdiv(a, b):
    return (a + b - 1) // b


def _cta(T, ch, S, sidx, t, accept_any_guess=False, no_lag=False):
    """Chunks a CTA scores, each with (rows scored, rows copied), or raises AssertionError."""
    spec_n = _cdiv(T - 1, ch)
    spec_c = sidx * _cdiv(spec_n, S)
    spec = spec_c < spec_n
    n_all = _cdiv(t, ch)
    per = _cdiv(n_all, S)
    k0 = sidx * per
    nck = max(0, min(n_all, k0 + per) - k0)
    spec_ok = spec and nck > 0 and (accept_any_guess or k0 == spec_c)
    lag = 1 if (spec and not spec_ok and not no_lag) else 0

    def chunk_of_fill(f):
        return k0 + f - lag if 0 <= f - lag < nck else -1

    fills = []  # fills[f] = (chunk or EMPTY or -1, rows copied)
    if spec:
        j0 = spec_c * ch
        fills.append((spec_c if spec_ok else EMPTY, min(T - 1, j0 + ch) - j0))
    while len(fills) < STAGES:
        c = chunk_of_fill(len(fills))
        fills.append((c, min(t, c * ch + ch) - c * ch if c >= 0 else 0))
    stage_phase = [0] * STAGES  # completed phases per stage (one per fill)
    for f in range(len(fills)):
        stage_phase[f % STAGES] += 1
    scored = []
    k = 0
    while True:
        st = k % STAGES
        # The consumer waits on parity (k / 3) & 1: the phase of fill k must have completed,
        # and the stage must not have run a further phase ahead of it.
        assert stage_phase[st] == k // STAGES + 1, "stage barrier phase out of step with the fill"
        c, copied = fills[k]
        if c == EMPTY:
            nf = len(fills)
            cc = chunk_of_fill(nf)
            fills.append((cc, min(t, cc * ch + ch) - cc * ch if cc >= 0 else 0))
            stage_phase[nf % STAGES] += 1
            k += 1
            continue
        if c < 0:
            break
        rc = min(t, c * ch + ch) - c * ch
        scored.append((c, rc, copied))
        nf = len(fills)
        cc = chunk_of_fill(nf)
        fills.append((cc, min(t, cc * ch + ch) - cc * ch if cc >= 0 else 0))
        stage_phase[nf % STAGES] += 1
        k += 1
        assert k <= nck + 2, "the consumer does not stop"
    return k0, nck, scored


def _check(T, ch, S, t, **kw):
    covered = []
    for sidx in range(S):
        k0, nck, scored = _cta(T, ch, S, sidx, t, **kw)
        assert [c for c, _, _ in scored] == list(range(k0, k0 + nck)), (T, ch, S, sidx, t, scored)
        for c, rc, copied in scored:
            assert 0 < rc <= copied, (T, ch, S, sidx, t, c, rc, copied)
            covered.extend(range(c * ch, c * ch + rc))
    assert covered == list(range(t)), (T, ch, S, t)


def _cases():
    for ch in (16, 64, 128):
        sizes = sorted({1, 2, 3, ch - 1, ch, ch + 1, ch + 2, 2 * ch, 2 * ch + 1, 3 * ch + 5, 8 * ch + 3})
        for T in sizes:
            if T < 1:
                continue
            for S in range(1, min(8, _cdiv(T, ch)) + 1):
                for t in range(T):
                    yield T, ch, S, t
    # The measured decode shapes (bf16 d 64: 128 rows; d 128: 64 rows), positions sampled.
    for T, ch in ((4096, 128), (16384, 64)):
        for S in (1, 2, 3, 5, 8):
            for t in (0, 1, ch - 1, ch, ch + 1, T // 2, T - ch - 1, T - ch, T - 2, T - 1):
                yield T, ch, S, t


def test_every_cta_scores_its_chunks_and_the_cluster_covers_the_cache():
    n = 0
    for T, ch, S, t in _cases():
        _check(T, ch, S, t)
        n += 1
    assert n > 10000


def test_planted_mistakes_are_caught():
    def fails(**kw):
        for T, ch, S, t in _cases():
            try:
                _check(T, ch, S, t, **kw)
            except AssertionError:
                return True
        return False

    assert fails(accept_any_guess=True)
    assert fails(no_lag=True)


def test_kernel_source_matches_the_model():
    src = open(os.path.join(CSRC, "decode.cu")).read()
    expect = [
        r"kStreamStages = 3;",
        r"spec_n = \(kp\.T - 1 \+ ch - 1\) / ch;",
        r"spec_c = sidx \* \(\(spec_n \+ S - 1\) / S\);",
        r"spec = spec_c < spec_n;",
        r"bytes = \(uint32_t\)\(\(min\(kp\.T - 1, j0 \+ ch\) - j0\) \* row_bytes\);",
        r"n_all = t_ok \? \(t \+ ch - 1\) / ch : 0;",
        r"per = \(n_all \+ S - 1\) / S;",
        r"k0 = sidx \* per;",
        r"nck = max\(0, min\(n_all, k0 \+ per\) - k0\);",
        r"spec_ok = spec && nck > 0 && k0 == spec_c;",
        r"lag = \(spec && !spec_ok\) \? 1 : 0;",
        r"chunk_of_fill = \[&\]\(int f\) \{ return \(f - lag >= 0 && f - lag < nck\) \? k0 \+ f - lag : -1; \};",
        r"int fills = spec \? 1 : 0;",
        r"mbar_wait\(&full\[st\], \(k / kStreamStages\) & 1,",
        r"if \(c == kEmptyStage\) \{",
        r"if \(c < 0\) break;",
    ]
    for e in expect:
        assert re.search(e, src), e
