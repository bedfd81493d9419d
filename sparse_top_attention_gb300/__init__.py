"""GB300-native sparse MLA (DSA) attention: forward and backward."""
