"""GB300-native target-verify path of tree-structured speculative decoding (placeholder; the
binding is added with the C-ABI library)."""
