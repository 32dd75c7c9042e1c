"""Masked token loss over packed labels. TEST INFRASTRUCTURE ONLY.

The XTuner page "序列并行" ("Sequence parallel", section "Reduce Loss"): the
model's loss on a rank is the mean token cross-entropy over the labels that
are not -100, num_tokens_per_rank = (labels != -100).sum(), and
reduce_sequence_parallel_loss combines the ranks' losses weighted by those
counts, so every rank ends with the loss of the whole sequence. The labels are
the pack's (InternEvo page "Data loading and flow": -100 at document ends and
padding).

Readings (listed in the design notes): cross-entropy of a token is
logsumexp(logits) - logits[label] (natural log); the loss of a set of tokens is
their sum divided by their count; a set with no counted token has loss 0; the
gradient with respect to the logits of a counted token is
(softmax(logits) - onehot(label)) * grad_scale (grad_scale = 1 / count for the
mean), 0 for an ignored token.

Plain fp64 numpy.
"""
import numpy as np

IGNORE_INDEX = -100


def token_losses(logits, labels):
    """[T, V] logits, [T] labels -> fp64 [T] cross-entropy, 0 where label == -100."""
    x = np.asarray(logits, dtype=np.float64)
    lab = np.asarray(labels)
    m = x.max(axis=1, keepdims=True)
    lse = (m + np.log(np.exp(x - m).sum(axis=1, keepdims=True)))[:, 0]
    out = np.zeros(x.shape[0])
    keep = lab != IGNORE_INDEX
    out[keep] = lse[keep] - x[keep, lab[keep]]
    return out


def masked_loss(logits, labels):
    """(sum of the counted tokens' losses, their count, mean or 0)."""
    lab = np.asarray(labels)
    s = float(token_losses(logits, labels).sum())
    n = int((lab != IGNORE_INDEX).sum())
    return s, n, (s / n if n else 0.0)


def reduce_sequence_parallel_loss(losses, counts):
    """Token-weighted combination of the ranks' mean losses."""
    n = sum(counts)
    return sum(l * c for l, c in zip(losses, counts)) / n if n else 0.0


def logits_grad(logits, labels, grad_scale):
    """(softmax - onehot) * grad_scale per counted token, 0 rows for ignored ones."""
    x = np.asarray(logits, dtype=np.float64)
    lab = np.asarray(labels)
    p = np.exp(x - x.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    keep = lab != IGNORE_INDEX
    rows = np.nonzero(keep)[0]
    p[rows, lab[keep]] -= 1.0
    p[~keep] = 0.0
    return p * grad_scale
