"""CPU oracle for exact full-context BPE tokenization (test infrastructure)."""
from .oracle import (  # noqa: F401
    Oracle, build_lib, load_class_table, class_table, byte_vocab, pretokenizer,
    FAMILY_CL100K_STYLE, FAMILY_O200K_STYLE, FAMILY_DEEPSEEK_STYLE, ERR_UTF8,
)
