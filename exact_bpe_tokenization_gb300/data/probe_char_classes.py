"""Write the frozen character-class table used by the pre-tokenizer.

The TokTier paper (arXiv 2607.29678, section 4.1 "run decomposition" and the
exactness discussion of section 5.2) pins the Unicode class tables by probing
them out of the reference regex engine instead of taking them from a library's
own Unicode data, because a Unicode-version skew between the two changed the
classes of ~9.7K code points.  This script does the same: it asks the installed
`regex` module, once per property, which scalar values match, and writes the
result as a range file with its SHA-256.

Properties probed (bit positions of the mask written per range):
    bit 0  \\p{L}     bit 1  \\p{Lu}    bit 2  \\p{Ll}    bit 3  \\p{Lt}
    bit 4  \\p{Lm}    bit 5  \\p{Lo}    bit 6  \\p{M}     bit 7  \\p{N}
    bit 8  \\s
Surrogates (U+D800..U+DFFF) are not scalar values and never reach the table's
users (UTF-8 decoding rejects them); they are written as mask 0.

Usage:  python probe_char_classes.py [out_path]
The file is committed; rerunning with the same `regex` release reproduces it
byte for byte (the test suite checks the stored SHA-256 and, where `regex` is
installed, re-probes and compares).
"""
import hashlib
import os
import sys

PROPS = [
    ("L", r"\p{L}"), ("Lu", r"\p{Lu}"), ("Ll", r"\p{Ll}"), ("Lt", r"\p{Lt}"),
    ("Lm", r"\p{Lm}"), ("Lo", r"\p{Lo}"), ("M", r"\p{M}"), ("N", r"\p{N}"),
    ("S", r"\s"),
]
MAX_CP = 0x110000


def probe_masks():
    """Return a list of MAX_CP ints: the property mask of every code point."""
    import regex  # the engine the table is frozen from

    masks = [0] * MAX_CP
    cps = [c for c in range(MAX_CP) if not (0xD800 <= c <= 0xDFFF)]
    text = "".join(chr(c) for c in cps)
    for bit, (_, pat) in enumerate(PROPS):
        for m in regex.finditer(pat, text):
            masks[ord(m.group())] |= 1 << bit
    return masks, regex.__version__


def masks_to_body(masks):
    lines = []
    start = 0
    for cp in range(1, MAX_CP + 1):
        if cp == MAX_CP or masks[cp] != masks[start]:
            if masks[start]:
                lines.append("%06X %06X %03X" % (start, cp - 1, masks[start]))
            start = cp
    return "\n".join(lines) + "\n"


def main(out_path):
    masks, version = probe_masks()
    body = masks_to_body(masks)
    digest = hashlib.sha256(body.encode("ascii")).hexdigest()
    header = (
        "# character classes probed from the regex engine, release %s\n"
        "# columns: first_cp last_cp mask (hex); bits L Lu Ll Lt Lm Lo M N \\s\n"
        "# code points not listed have mask 0\n"
        "# body-sha256 %s\n" % (version, digest)
    )
    with open(out_path, "w", encoding="ascii") as f:
        f.write(header + body)
    print(out_path, digest)


if __name__ == "__main__":
    here = os.path.dirname(os.path.abspath(__file__))
    main(sys.argv[1] if len(sys.argv) > 1 else os.path.join(here, "char_classes.txt"))
