"""Seeded synthetic inputs: transcript text, adversarial text, request lengths
and greedy-trained merge lists.  Inputs only; no tokenizer arithmetic."""
from .synth import (  # noqa: F401
    PROFILE_ASCII, PROFILE_MIXED, PROFILE_CAMEL_MARKS, PROFILE_KANA_HAN, FAMILY_DEEPSEEK_STYLE,
    build_lib, transcript, adversarial, lengths_loguniform, lengths_lognormal,
    train_merges, vocab_from_merges, make_vocab, batch, WORKLOADS, workload,
)
